"""The bounded mbarrier wait of the decode kernels, made to run out.

Every wait in the library's kernels goes through `pkv::mbar_wait`
(csrc/pkv_common.cuh), which gives up after a time limit (2 s by default) and
returns false; the kernel then sets PKV_DEVERR_TIMEOUT and stops instead of
hanging.  The kernels' own waits can only run out on a copy that never lands,
which no test may cause.  So this test builds a small kernel of its own around
the same primitive: one CTA initialises an mbarrier, issues no copy at all and
waits on a phase nothing will complete, with a 1 ms limit.  Nothing is in flight,
so the kernel ends by itself; the test checks that the wait reported failure,
that it waited at least its limit and not much longer, that the timeout bit was
set, and that the context is still usable afterwards.
"""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

SRC = r'''
#include "pkv_common.cuh"

__global__ void wait_on_nothing(unsigned long long limit_ns, unsigned int* flags,
                                unsigned long long* waited_ns) {
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t b = pkv::smem_addr(&bar);
    if (threadIdx.x == 0) {
        pkv::mbar_init(b, 1);
        pkv::mbar_init_fence();
    }
    __syncthreads();
    const unsigned long long t0 = pkv::global_ns();
    const bool done = pkv::mbar_wait(b, 0, limit_ns);   // phase 0: nothing ever arrives
    const unsigned long long t1 = pkv::global_ns();
    if (!done) pkv::set_error(&flags[0], PKV_DEVERR_TIMEOUT);
    if (done) atomicAdd(&flags[1], 1u);                   // lanes whose wait claimed success
    if (threadIdx.x == 0) waited_ns[0] = t1 - t0;
}

extern "C" int run_wait(unsigned long long limit_ns, unsigned int* flags_out,
                        unsigned long long* waited_out) {
    unsigned int* flags = nullptr;
    unsigned long long* waited = nullptr;
    if (cudaMalloc(&flags, 2 * sizeof(unsigned int)) != cudaSuccess) return 1;
    if (cudaMalloc(&waited, sizeof(unsigned long long)) != cudaSuccess) return 2;
    cudaMemset(flags, 0, 2 * sizeof(unsigned int));
    wait_on_nothing<<<1, 32>>>(limit_ns, flags, waited);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(flags_out, flags, 2 * sizeof(unsigned int),
                                         cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(waited_out, waited, sizeof(unsigned long long),
                                         cudaMemcpyDeviceToHost);
    cudaFree(flags);
    cudaFree(waited);
    return e == cudaSuccess ? 0 : 100 + (int)e;
}
'''


@pytest.fixture(scope="module")
def waitlib(tmp_path_factory):
    from paged_kv_cache_293_gb300 import _build
    d = tmp_path_factory.mktemp("waitkernel")
    src = d / "wait_kernel.cu"
    src.write_text(SRC)
    so = d / "libwait.so"
    cmd = [_build.nvcc(), *_build.ARCH, *_build.NVCC_FLAGS, "-I" + _build.CSRC, "-shared",
           str(src), "-o", str(so)]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    assert proc.returncode == 0, proc.stderr
    lib = ctypes.CDLL(str(so))
    lib.run_wait.argtypes = [ctypes.c_ulonglong, ctypes.POINTER(ctypes.c_uint),
                             ctypes.POINTER(ctypes.c_ulonglong)]
    lib.run_wait.restype = ctypes.c_int
    return lib


def test_wait_on_an_mbarrier_nothing_arrives_on_gives_up_at_its_limit(waitlib):
    from paged_kv_cache_293_gb300 import pagedkv as P
    torch.cuda.init()
    limit_ns = 1_000_000                                   # 1 ms
    flags = (ctypes.c_uint * 2)()
    waited = ctypes.c_ulonglong()
    rc = waitlib.run_wait(limit_ns, flags, ctypes.byref(waited))
    assert rc == 0, "CUDA error %d" % rc
    assert flags[0] == P.DEVERR["TIMEOUT"]                 # every lane gave up and flagged it
    assert flags[1] == 0                                   # no lane claimed the phase completed
    assert limit_ns <= waited.value < limit_ns + 50_000_000, waited.value
    # the context is still usable: a plain torch kernel runs after it
    x = torch.arange(4, device="cuda")
    assert int((x * 2).sum()) == 12
