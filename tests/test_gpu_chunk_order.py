"""The order in which a warp of the tensor-core decode kernel walks its chunks.

`pkv::alternating_chunk(i, n)` (csrc/pkv_common.cuh) gives the position, in the
warp's own list of n chunks, of the chunk it handles at step i: 0, n-1, 1, n-2,
...  Every chunk must be handled exactly once, whatever n.  A one-CTA kernel built
here evaluates the library's own device function for every n up to 2048 and the
host checks that each row is a permutation with the stated pattern.
"""
import ctypes
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

NMAX = 2048

SRC = r'''
#include "pkv_common.cuh"

__global__ void orders(int nmax, int* out) {
    for (int n = blockIdx.x; n <= nmax; n += gridDim.x)
        for (int i = threadIdx.x; i < n; i += blockDim.x)
            out[(size_t)n * nmax + i] = pkv::alternating_chunk(i, n);
}

extern "C" int run_orders(int nmax, int* host_out) {
    int* d = nullptr;
    const size_t bytes = (size_t)(nmax + 1) * nmax * sizeof(int);
    if (cudaMalloc(&d, bytes) != cudaSuccess) return 1;
    cudaMemset(d, 0xff, bytes);
    orders<<<64, 256>>>(nmax, d);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaMemcpy(host_out, d, bytes, cudaMemcpyDeviceToHost);
    cudaFree(d);
    return e == cudaSuccess ? 0 : 100 + (int)e;
}
'''


@pytest.fixture(scope="module")
def orderlib(tmp_path_factory):
    from paged_kv_cache_293_gb300 import _build
    d = tmp_path_factory.mktemp("chunkorder")
    src = d / "chunk_order.cu"
    src.write_text(SRC)
    so = d / "liborder.so"
    cmd = [_build.nvcc(), *_build.ARCH, *_build.NVCC_FLAGS, "-I" + _build.CSRC, "-shared",
           str(src), "-o", str(so)]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    assert proc.returncode == 0, proc.stderr
    lib = ctypes.CDLL(str(so))
    lib.run_orders.argtypes = [ctypes.c_int, ctypes.c_void_p]
    lib.run_orders.restype = ctypes.c_int
    return lib


def test_alternating_chunk_order_visits_every_chunk_once(orderlib):
    out = np.empty((NMAX + 1) * NMAX, dtype=np.int32)
    rc = orderlib.run_orders(NMAX, out.ctypes.data)
    assert rc == 0, "CUDA error %d" % rc
    out = out.reshape(NMAX + 1, NMAX)
    for n in range(NMAX + 1):
        row = out[n, :n]
        assert np.array_equal(np.sort(row), np.arange(n)), n
        # front and back alternately: steps 0, 2, 4, ... count up from 0, steps 1, 3, ... down
        assert np.array_equal(row[0::2], np.arange(len(row[0::2]))), n
        assert np.array_equal(row[1::2], n - 1 - np.arange(len(row[1::2]))), n
