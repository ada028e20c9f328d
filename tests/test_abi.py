"""The C-ABI library loads and exports every symbol include/sf.h declares;
host-side logic that needs no GPU (sizes, validation, RoPE table)."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

import inputs
from inputs import CONFIGS, UNIT_EMBED, UNIT_FINAL_NORM, UNIT_LM_HEAD

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "sf.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sf_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def sf():
    import offloaded_fine_tuning_gb300 as sfp
    return sfp.lib(build_if_needed=True), sfp


def test_library_exports_every_declared_symbol(sf):
    L, sfp = sf
    names = header_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(sfp.exported_names())


def test_unit_numel_matches_shapes(sf):
    _, sfp = sf
    for c in CONFIGS.values():
        cfg = sfp.make_config(c)
        for u in (0, UNIT_EMBED, UNIT_FINAL_NORM, UNIT_LM_HEAD):
            assert sfp.unit_numel(cfg, u) == inputs.unit_numel(c, u)
        assert sfp.unit_numel(cfg, c.n_layers) == 0 and sfp.unit_numel(cfg, -4) == 0


@pytest.mark.parametrize("field,value", [("head_dim", 96), ("n_kv_heads", 3), ("hidden", 100),
                                         ("vocab", 1001), ("ring_slots", 1), ("max_seq", 0)])
def test_invalid_config_rejected_before_any_cuda_call(sf, field, value):
    L, sfp = sf
    cfg = sfp.make_config(CONFIGS["tiny"])
    setattr(cfg, field, value)
    h = ctypes.c_void_p()
    assert L.sf_init_model(ctypes.byref(cfg), ctypes.byref(h)) == sfp.SF_EINVAL
    assert not h.value
    assert len(L.sf_last_error(None)) > 0


def test_rope_table_values(sf):
    _, sfp = sf
    t = sfp.rope_table(50, 128, 500000.0)
    j = np.arange(64)
    ang = np.arange(50)[:, None] * 500000.0 ** (-2.0 * j / 128)[None, :]
    assert np.allclose(t[..., 0], np.cos(ang), atol=1e-7) and np.allclose(t[..., 1], np.sin(ang), atol=1e-7)
    assert t[0, :, 0].min() == 1.0 and not t[0, :, 1].any()


def test_kernel_api_rejects_bad_arguments_without_launching(sf):
    _, sfp = sf
    # misaligned / null operands and bad sizes are refused on the host
    assert sfp.op_gemm(sfp.NT, sfp.EPI_BF16, 10, 10, 10, 8, 10, 0, 10, 0, 10) == sfp.SF_EINVAL
    assert sfp.op_gemm(7, 0, 1, 1, 1, 0, 1, 0, 1, 0, 1) == sfp.SF_EINVAL
    assert sfp.op_attn_fwd(0, 0, 0, 1, 16, 4, 3, 64) == sfp.SF_EINVAL
    assert sfp.op_rmsnorm_fwd(16, 16, 16, 16, 1, 16392, 1e-5) == sfp.SF_EINVAL  # d above 16384
    assert sfp.op_attn_fwd(0, 0, 0, 1, 16, 4, 2, 96) == sfp.SF_EINVAL
    assert sfp.op_swiglu_fwd(0, 0, 4, 12) == sfp.SF_EINVAL
    assert sfp.lce_workspace_bytes(100, 1000, 64) >= 64 * 1000 * 2 + 400
    # the workspace holds a chunk's fp32 logits and bf16 dZ, 256-aligned, then the row losses
    r256 = lambda x: (x + 255) // 256 * 256
    assert sfp.lce_workspace_bytes(100, 1000, 64) == r256(4 * 64 * 1000) + r256(2 * 64 * 1000) + r256(4 * 100)
    assert sfp.lce_workspace_bytes(50, 1000, 64) == r256(4 * 50 * 1000) + r256(2 * 50 * 1000) + r256(4 * 50)
    # sf_op_lce: vocabulary not a multiple of 8, misaligned workspace, n_valid above n
    a = 4096
    assert sfp.op_lce(a, a, a, 16, 64, 1004, 16, 16, a, a, a, a) == sfp.SF_EINVAL
    assert sfp.op_lce(a, a, a, 16, 64, 1000, 16, 16, a + 16, a, a, a) == sfp.SF_EINVAL
    assert sfp.op_lce(a, a, a, 16, 64, 1000, 17, 16, a, a, a, a) == sfp.SF_EINVAL
    assert sfp.lce_launches() == 0  # no call has launched anything on this thread
