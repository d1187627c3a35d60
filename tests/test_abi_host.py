"""CPU-only checks of the C ABI: the library loads, exports every entry point
declared in include/mtgr.h, and rejects bad scalar arguments on the host
(before any CUDA call, so no GPU is needed)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "mtgr.h")).read()
    return sorted(set(re.findall(r"MTGR_API\s+[\w\s\*]*?\b(mtgr_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from hstu_attention_attn_b300 import build, mtgr
    build.build()
    return mtgr.lib()


def test_header_declares_entry_points():
    names = _declared()
    for n in ("mtgr_group_layernorm_fwd", "mtgr_group_layernorm_bwd", "mtgr_hstu_attn_fwd", "mtgr_hstu_attn_bwd",
              "mtgr_hstu_layer_fwd", "mtgr_hstu_layer_bwd", "mtgr_validate_batch", "mtgr_debug_visible_counts"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared():
        assert hasattr(lib, n), f"libmtgr.so does not export {n}"


def test_binding_covers_every_symbol():
    from hstu_attention_attn_b300 import mtgr
    for n in _declared():
        assert n in mtgr.EXPORTS and hasattr(mtgr, n), n


def test_version_and_workspace_queries(lib):
    from hstu_attention_attn_b300 import mtgr
    assert mtgr.mtgr_version() >= 100
    a = mtgr.mtgr_attn_workspace_size(64, 47000, 4, 128, mtgr.MTGR_BF16)
    b = mtgr.mtgr_attn_workspace_size(64, 94000, 4, 128, mtgr.MTGR_BF16)
    assert 0 < a < b
    assert mtgr.mtgr_attn_workspace_size(-1, 10, 4, 128, mtgr.MTGR_BF16) == 0
    assert mtgr.mtgr_layer_workspace_size(128, 63000, 1024, 8, 128, mtgr.MTGR_BF16) > 0


def test_bad_scalars_rejected_on_host(lib):
    from hstu_attention_attn_b300 import mtgr
    L = mtgr.lib()
    # D not a multiple of 8 -> unsupported, no CUDA call made
    r = L.mtgr_group_layernorm_fwd(None, None, None, None, None, None, None, 10, 7, 1e-5, mtgr.MTGR_BF16, None)
    assert r == -4 and "multiple of 8" in mtgr.mtgr_last_error()
    # bf16 attention with d_h = 96 -> unsupported
    r = L.mtgr_hstu_attn_fwd(None, None, None, None, 384, None, 1, None, None, 10, 4, 96, 1e-5, None, None, None,
                             None, mtgr.MTGR_BF16, None, 0, None)
    assert r in (-1, -4)
    # missing workspace
    r = L.mtgr_hstu_attn_fwd(16, 16, 16, 16, 512, 16, 1, 16, 16, 10, 4, 128, 1e-5, 16, 16, 16, 16,
                             mtgr.MTGR_BF16, None, 0, None)
    assert r == -7
    # negative sizes
    r = L.mtgr_validate_batch(16, -1, 16, 10, 16, None)
    assert r == -1


def test_expand_rows_rejects_bad_arguments_on_the_host(lib):
    import ctypes as C
    from hstu_attention_attn_b300 import mtgr
    buf = (C.c_uint8 * 4096)()
    p = C.addressof(buf) + (-C.addressof(buf)) % 16          # a 16-byte aligned host address, never read
    # D = 7 bf16 values is not a multiple of 16 bytes
    assert lib.mtgr_expand_rows(p, p, 1, p, 4, 7, mtgr.MTGR_BF16, None) == mtgr.MTGR_ERR_INVALID_ARG
    assert lib.mtgr_expand_rows(None, None, 1, p, 4, 8, mtgr.MTGR_BF16, None) == mtgr.MTGR_ERR_INVALID_ARG
    assert lib.mtgr_expand_rows(p, p, -1, p, 4, 8, mtgr.MTGR_BF16, None) == mtgr.MTGR_ERR_INVALID_ARG


def test_plan_counts_rejects_bad_arguments_on_the_host(lib):
    import ctypes as C
    from hstu_attention_attn_b300 import mtgr
    out = (C.c_int32 * 4)()
    assert lib.mtgr_debug_plan_counts(None, 4, out, None) == mtgr.MTGR_ERR_INVALID_ARG
    assert lib.mtgr_debug_plan_counts(C.addressof(out), 4, None, None) == mtgr.MTGR_ERR_INVALID_ARG
    assert lib.mtgr_debug_plan_counts(C.addressof(out), -1, out, None) == mtgr.MTGR_ERR_INVALID_ARG


def test_wait_timeout_check_rejects_null_status(lib):
    from hstu_attention_attn_b300 import mtgr
    assert lib.mtgr_debug_wait_timeout(None, None) == mtgr.MTGR_ERR_INVALID_ARG
    assert "status_word" in mtgr.mtgr_last_error()


def test_binding_refuses_host_tensors(lib):
    import torch
    from hstu_attention_attn_b300 import mtgr
    assert mtgr._p(None) is None and mtgr._p(4096) == 4096
    with pytest.raises(ValueError, match="CUDA tensor"):
        mtgr._p(torch.zeros(4))
    st = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        mtgr.mtgr_validate_batch(torch.zeros(2, dtype=torch.int32), torch.zeros(1, dtype=torch.uint8), 1, st, stream=0)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """There is no CPU fallback: without libmtgr.so every entry point raises."""
    import torch
    from hstu_attention_attn_b300 import mtgr
    monkeypatch.setattr(mtgr, "LIB_PATH", str(tmp_path / "libmtgr.so"))
    monkeypatch.setattr(mtgr, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        mtgr.lib()
    with pytest.raises(RuntimeError, match="missing"):
        mtgr.mtgr_version()
    with pytest.raises(RuntimeError, match="missing"):
        mtgr.mtgr_token_balanced_split([3, 4, 5], 2)


def test_ds_store_size_query(lib):
    """Bytes of the backward's dS tile store: one 128 x 128 f16 tile per head
    and per cell of each user's (query tile, key tile) grid, plus 1024 bytes
    of alignment; 0 where the store is not used.  Host memory only."""
    import numpy as np
    from hstu_attention_attn_b300 import mtgr
    rng = np.random.default_rng(5)
    lens = np.concatenate([[0, 1, 127, 128, 129, 256, 1092], rng.integers(0, 3000, 50)])
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    grid = sum(((int(n) + 127) // 128) ** 2 for n in lens)
    for H, dh in ((8, 128), (2, 64)):
        assert mtgr.mtgr_attn_ds_store_size(offs, H, dh, mtgr.MTGR_BF16) == H * grid * 32768 + 1024
    assert mtgr.mtgr_attn_ds_store_size(offs, 8, 128, mtgr.MTGR_F32) == 0
    assert mtgr.mtgr_attn_ds_store_size(offs, 8, 32, mtgr.MTGR_BF16) == 0
    assert mtgr.mtgr_attn_ds_store_size(offs, 0, 128, mtgr.MTGR_BF16) == 0
    assert mtgr.mtgr_attn_ds_store_size(np.array([0, 0, 0], np.int32), 8, 128, mtgr.MTGR_BF16) == 0
    assert mtgr.mtgr_attn_ds_store_size(np.array([0, 300, 200], np.int32), 8, 128, mtgr.MTGR_BF16) == 0
