"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every
function include/moe_nvfp4.h declares, its structs have the ctypes layout the
binding uses, and host-side validation (default-deny configuration checks,
argument checks) answers before any CUDA work."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_nvfp4.h")


@pytest.fixture(scope="module")
def moe():
    from nvfp4_weight_only_fp32_gb300 import build
    build.build()
    import nvfp4_weight_only_fp32_gb300 as m
    m.lib()
    return m


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(moe):
    names = declared_functions()
    assert len(names) >= 12
    L = moe.lib()
    for n in names:
        assert hasattr(L, n), n
    assert sorted(moe.EXPORTED) == names
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True, text=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}\b", out), n


def test_struct_layout_matches_header(moe, tmp_path):
    prog = tmp_path / "layout.c"
    prog.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "moe_nvfp4.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\n", sizeof(moe_config), sizeof(moe_weights), sizeof(moe_layer_info),
         offsetof(moe_config, routed_scale), offsetof(moe_config, grouped_min_tokens),
         offsetof(moe_weights, sw2_gs), offsetof(moe_layer_info, sm_count),
         offsetof(moe_config, fused), offsetof(moe_layer_info, single_launch_max_tokens),
         offsetof(moe_config, score_func), offsetof(moe_config, expert_format), offsetof(moe_config, w4a4));
  return 0; }
''')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()]
    want = [ctypes.sizeof(moe.moe_config), ctypes.sizeof(moe.moe_weights),
            ctypes.sizeof(moe.moe_layer_info), moe.moe_config.routed_scale.offset,
            moe.moe_config.grouped_min_tokens.offset, moe.moe_weights.sw2_gs.offset,
            moe.moe_layer_info.sm_count.offset, moe.moe_config.fused.offset,
            moe.moe_layer_info.single_launch_max_tokens.offset, moe.moe_config.score_func.offset,
            moe.moe_config.expert_format.offset, moe.moe_config.w4a4.offset]
    assert got == want


def _cfg(moe, **kw):
    base = dict(hidden=2048, num_experts=256, top_k=6, inter=768, num_shared=1, shared_inter=768,
                max_tokens=8, normalize_topk=1, routed_scale=1.0, grouped_min_tokens=0, fused=0)
    base.update(kw)
    return moe.moe_config(**base)


def test_default_deny_lists_every_reason(moe):
    L = moe.lib()
    h = ctypes.c_void_p()
    bad = _cfg(moe, hidden=100, inter=0, top_k=9, max_tokens=65, num_shared=3, score_func=2, w4a4=2)
    rc = L.moe_init(ctypes.byref(bad), ctypes.byref(moe.moe_weights()), None, ctypes.byref(h))
    assert rc == moe.moe.MOE_ERR_UNSUPPORTED
    msg = moe.last_error()
    for frag in ("hidden", "inter", "top_k", "max_tokens", "num_shared", "score_func", "w4a4"):
        assert frag in msg, (frag, msg)
    assert not h.value


def test_null_and_host_pointers_rejected(moe):
    L = moe.lib()
    h = ctypes.c_void_p()
    rc = L.moe_init(ctypes.byref(_cfg(moe)), ctypes.byref(moe.moe_weights()), None, ctypes.byref(h))
    assert rc == moe.moe.MOE_ERR_INVALID_ARG
    assert "router_w is NULL" in moe.last_error()
    buf = ctypes.create_string_buffer(64)          # host memory, not a device pointer
    addr = (ctypes.addressof(buf) + 15) // 16 * 16
    w = moe.moe_weights(**{n: addr for n, _ in moe.moe_weights._fields_})
    rc = L.moe_init(ctypes.byref(_cfg(moe)), ctypes.byref(w), None, ctypes.byref(h))
    assert rc == moe.moe.MOE_ERR_INVALID_ARG
    assert "not a device pointer" in moe.last_error()


def test_calls_on_null_handle(moe):
    L = moe.lib()
    assert L.moe_decode_forward(None, None, 1, None, None, None, None) == moe.moe.MOE_ERR_INVALID_ARG
    assert L.moe_stage_down(None, 1, None, None) == moe.moe.MOE_ERR_INVALID_ARG
    assert L.moe_check(None, None) == moe.moe.MOE_ERR_INVALID_ARG
    assert L.moe_get_info(None, None) == moe.moe.MOE_ERR_INVALID_ARG
    L.moe_destroy(None)


def test_quantiser_arguments_checked_before_any_launch(moe):
    L = moe.lib()
    assert L.moe_quant_fos(None, 2, 24, None, None, None) == moe.moe.MOE_ERR_INVALID_ARG
    assert "multiple of 16" in moe.last_error()
    assert L.moe_quant_fos(None, -1, 32, None, None, None) == moe.moe.MOE_ERR_INVALID_ARG
    assert L.moe_quant_fos(None, 1, 32, None, None, None) == moe.moe.MOE_ERR_INVALID_ARG
    assert "NULL" in moe.last_error()
    assert L.moe_quant_fos(None, 0, 32, None, None, None) == moe.moe.MOE_OK    # nothing to do
    # a pointer off the 8-byte grid is refused before anything touches it
    assert L.moe_quant_fos(0x1004, 1, 32, 0x2000, 0x3000, None) == moe.moe.MOE_ERR_INVALID_ARG
    assert "8-byte aligned" in moe.last_error()
