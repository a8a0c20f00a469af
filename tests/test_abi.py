"""The C-ABI library builds, loads and exports every function include/pagedkv.h
declares; host-side argument checks answer before any CUDA call (CPU only)."""
import ctypes
import shutil

import pytest
import torch

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and
                                not __import__("os").path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


@pytest.fixture(scope="module")
def P():
    from paged_kv_cache_293_gb300 import _build
    _build.build()
    from paged_kv_cache_293_gb300 import pagedkv
    return pagedkv


def test_every_declared_function_is_exported(P):
    names = P.declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(P.lib, n), n
    # and the binding wraps each one under the same name
    import paged_kv_cache_293_gb300.pagedkv as mod
    for n in names:
        assert callable(getattr(mod, n)), n


def test_version_and_status_text(P):
    assert P.pkv_version() >= 100
    assert P.pkv_status_str(P.PKV_OK) == "ok"
    assert "workspace" in P.pkv_status_str(P.PKV_ERR_WORKSPACE)


def _pool(**kw):
    d = dict(k=16, v=32, num_blocks=4, block_size=16, num_kv_heads=2, head_dim=128, dtype=1)
    d.update(kw)
    from paged_kv_cache_293_gb300.pagedkv import pkv_pool
    return pkv_pool(d["k"], d["v"], d["num_blocks"], d["block_size"], d["num_kv_heads"],
                    d["head_dim"], d["dtype"])


def _decode(P, pool, S=1, Hq=2, M=4, max_ctx=10, P_=0, out_dtype=1, scale=0.1, ws=None,
            ws_bytes=0, ptrs=True):
    dummy = ctypes.c_void_p(256) if ptrs else None
    return P.lib.pkv_paged_attention_decode(ctypes.byref(pool) if pool is not None else None,
                                            dummy, S, Hq, dummy, M, dummy, max_ctx, scale, dummy,
                                            out_dtype, P_, ws, ws_bytes, None)


def test_decode_argument_checks(P):
    assert _decode(P, None) == P.PKV_ERR_INVALID
    assert _decode(P, _pool(k=0)) == P.PKV_ERR_INVALID
    assert _decode(P, _pool(k=8)) == P.PKV_ERR_INVALID               # misaligned
    assert _decode(P, _pool(dtype=7)) == P.PKV_ERR_INVALID
    assert _decode(P, _pool(block_size=8)) == P.PKV_ERR_UNSUPPORTED
    assert _decode(P, _pool(head_dim=96)) == P.PKV_ERR_UNSUPPORTED
    assert _decode(P, _pool(), Hq=3) == P.PKV_ERR_INVALID            # Hq % Hkv
    assert _decode(P, _pool(num_kv_heads=1), Hq=16) == P.PKV_ERR_UNSUPPORTED  # group 16
    assert _decode(P, _pool(), P_=24) == P.PKV_ERR_INVALID           # not a multiple of B
    assert _decode(P, _pool(), out_dtype=2) == P.PKV_ERR_UNSUPPORTED  # bf16 out of an fp16 pool
    assert _decode(P, _pool(), scale=float("nan")) == P.PKV_ERR_INVALID
    assert _decode(P, _pool(), ptrs=False) == P.PKV_ERR_INVALID
    assert _decode(P, _pool(), max_ctx=5000, P_=512) == P.PKV_ERR_WORKSPACE
    assert _decode(P, _pool(), S=0) == P.PKV_OK                      # nothing to do
    assert _decode(P, _pool(), S=65536) == P.PKV_ERR_UNSUPPORTED     # one grid row per sequence


def test_cascade_argument_checks(P):
    d = ctypes.c_void_p(256)

    def call(pool, prefix=32, max_ctx=100, kn=None, vn=None, ws=d, ws_bytes=1 << 30, S=2):
        return P.lib.pkv_paged_attention_decode_cascade(
            ctypes.byref(pool), d, S, 2, d, 16, d, max_ctx, 0.1, prefix, d, 0, 0, kn, vn, None,
            ws, ws_bytes, None)

    assert call(_pool(dtype=0)) == P.PKV_ERR_UNSUPPORTED                  # fp32 pool
    assert call(_pool(), prefix=24) == P.PKV_ERR_INVALID                  # not a multiple of 16
    assert call(_pool(), prefix=0) == P.PKV_ERR_INVALID
    assert call(_pool(), prefix=112) == P.PKV_ERR_INVALID                 # past max_context_len
    assert call(_pool(), kn=d) == P.PKV_ERR_INVALID                       # k_new without v_new
    assert call(_pool(), ws=None) == P.PKV_ERR_WORKSPACE
    assert call(_pool(), ws_bytes=16) == P.PKV_ERR_WORKSPACE
    # 2^32 (block, kv head, position) rows: past the tensor maps' int32 rows, refused
    # before any launch
    assert call(_pool(num_blocks=1 << 27)) == P.PKV_ERR_UNSUPPORTED
    f = P.lib.pkv_cascade_workspace_bytes
    assert f(ctypes.byref(_pool()), 2, 2, 100, 32, 0) > 0


def test_multi_query_append_argument_checks(P):
    d = ctypes.c_void_p(256)

    def call(pool, kn=d, vn=d, nq=4, S=1, out_dtype=1):
        return P.lib.pkv_paged_attention_decode_multi_append(
            ctypes.byref(pool), d, kn, vn, nq, S, 2, d, 4, d, 10, 0.1, d, out_dtype, 0, None, 0,
            None, None)

    assert call(_pool(), kn=None) == P.PKV_ERR_INVALID
    assert call(_pool(), vn=ctypes.c_void_p(8)) == P.PKV_ERR_INVALID      # misaligned rows
    assert call(_pool(), nq=0) == P.PKV_ERR_INVALID
    assert call(_pool(dtype=0), out_dtype=0) == P.PKV_ERR_UNSUPPORTED     # fp32 pool
    assert call(_pool(), out_dtype=2) == P.PKV_ERR_UNSUPPORTED            # bf16 out, fp16 pool
    assert call(_pool(), S=65536) == P.PKV_ERR_UNSUPPORTED
    assert call(_pool(), S=0) == P.PKV_OK


def test_workspace_sizes(P):
    pool = _pool()
    f = P.lib.pkv_decode_workspace_bytes
    assert f(ctypes.byref(pool), 8, 32, 512, 512) == 0               # one pass
    rows = 8 * 32 * 2
    a = (rows * 4 + 15) // 16 * 16
    assert f(ctypes.byref(pool), 8, 32, 1000, 512) == 2 * a + rows * 128 * 4
    assert P.lib.pkv_partition_workspace_bytes(8, 32, 128, 100, 512) == 2 * ((8 * 32 * 4 + 15) // 16 * 16) + 8 * 32 * 128 * 4
    assert P.lib.pkv_choose_partition_size(ctypes.byref(pool), 8, 32, 100) % 16 == 0


def test_other_entry_points_check_arguments(P):
    pool = _pool()
    d = ctypes.c_void_p(256)
    assert P.lib.pkv_kv_cache_write(None, d, d, d, 1, None) == P.PKV_ERR_INVALID
    assert P.lib.pkv_kv_cache_write(ctypes.byref(pool), d, d, d, 0, None) == P.PKV_OK
    assert P.lib.pkv_kv_cache_write(ctypes.byref(pool), ctypes.c_void_p(8), d, d, 1, None) == P.PKV_ERR_INVALID
    assert P.lib.pkv_copy_blocks(ctypes.byref(pool), None, 3, None) == P.PKV_ERR_INVALID
    assert P.lib.pkv_copy_blocks(ctypes.byref(pool), d, 0, None) == P.PKV_OK
    assert P.lib.pkv_slot_mapping(d, 4, 2, d, None, 0, 16, d, None) == P.PKV_OK
    assert P.lib.pkv_slot_mapping(d, 4, 2, d, None, 3, 16, d, None) == P.PKV_ERR_INVALID
    assert P.lib.pkv_slot_mapping(None, 4, 2, d, None, 1, 16, d, None) == P.PKV_ERR_INVALID
    assert P.lib.pkv_lse_merge(None, 0, 1, 8, 128, d, 10, 16, d, 0, None) == P.PKV_ERR_WORKSPACE
    assert P.lib.pkv_lse_merge(d, 1 << 20, 1, 8, 96, d, 10, 16, d, 0, None) == P.PKV_ERR_UNSUPPORTED
    assert P.lib.pkv_get_device_error(None, None) == P.PKV_ERR_INVALID


def test_binding_rejects_non_contiguous_tensors(P):
    k = torch.zeros(4, 2, 16, 128, dtype=torch.float16).transpose(1, 2)
    with pytest.raises(ValueError):
        P.make_pool(k, k)
