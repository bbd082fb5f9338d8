"""The quantiser's division (div_by_recip in csrc/qevict_div.cuh: the rounded
reciprocal of the scale and one FMA correction, Markstein 1990) against a
correctly rounded fp32 division: bit for bit wherever the quotient is a normal
fp32 number, and to the same integer code (zero) where it is subnormal, which
the correction step does not cover. Divisors: every positive finite
fp16 value (normal and subnormal), as the quantiser's scales are. Dividends:
for each divisor, the fp32 values within four ulps of n * b and (n + 1/2) * b
for n = 0..255 (the rounding boundaries that decide an 8-bit code) and 512
pseudo-random values in [-b, 260 b]. The kernel compiles the library's own
header, so it checks the code the quantiser runs."""
import ctypes
import os
import subprocess
import tempfile

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "tiered_kv_cache_decode_gb300", "csrc")

_SRC = r"""
#include <cuda_fp16.h>
#include <stdint.h>
#include "qevict_div.cuh"

__device__ float step_ulps(float x, int k) {   // k ulps away in fp32 (x finite, nonzero steps stay finite)
    int32_t i = __float_as_int(x);
    if (x == 0.f) return k == 0 ? 0.f : __int_as_float(k > 0 ? k : (0x80000000 | -k));
    if (i < 0) k = -k;
    return __int_as_float(i + k);
}

__device__ void check(float a, float b, float rb, unsigned long long *bad, float *first) {
    const float q = qevict::div_by_recip(a, b, rb);
    const float ref = __fdiv_rn(a, b);
    // a normal quotient must match bit for bit; a subnormal one (|a| below 2^-126 b)
    // only has to round to the same integer code (zero)
    const bool normal = fabsf(ref) >= 1.17549435e-38f;
    const bool same = normal ? __float_as_int(q) == __float_as_int(ref) : fabsf(rintf(q)) == fabsf(rintf(ref));
    if (!same) {
        if (atomicAdd(bad, 1ull) == 0ull) {
            first[0] = a;
            first[1] = b;
            first[2] = q;
            first[3] = ref;
        }
    }
}

// blockIdx.x: fp16 divisor bits 1 .. 0x7bff; thread: dividends
__global__ void div_kernel(unsigned long long *bad, float *first) {
    const unsigned short hb = (unsigned short)(blockIdx.x + 1);
    const float b = __half2float(__ushort_as_half(hb));
    const float rb = __frcp_rn(b);
    for (int it = threadIdx.x; it < 256 * 2 * 9; it += blockDim.x) {
        const int n = it / 18, r = it % 18, half = r / 9, k = r % 9 - 4;
        const float base = __fmul_rn(half ? (float)n + 0.5f : (float)n, b);
        check(step_ulps(base, k), b, rb, bad, first);
    }
    for (int it = threadIdx.x; it < 512; it += blockDim.x) {
        uint32_t h = (uint32_t)hb * 2654435761u ^ (uint32_t)it * 2246822519u;
        h ^= h >> 15; h *= 2246822519u; h ^= h >> 13; h *= 3266489917u; h ^= h >> 16;
        const float u = (float)(h >> 8) * (1.f / 16777216.f);   // [0, 1)
        check(__fmul_rn(__fmaf_rn(u, 261.f, -1.f), b), b, rb, bad, first);
    }
}

extern "C" int run_div_check(unsigned long long *bad_host, float *first_host) {
    unsigned long long *bad;
    float *first;
    if (cudaMalloc(&bad, 8) != cudaSuccess || cudaMalloc(&first, 16) != cudaSuccess) return -1;
    cudaMemset(bad, 0, 8);
    cudaMemset(first, 0, 16);
    div_kernel<<<0x7bff, 256>>>(bad, first);
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(bad_host, bad, 8, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(first_host, first, 16, cudaMemcpyDeviceToHost);
    cudaFree(bad);
    cudaFree(first);
    return (int)e;
}
"""


def test_quantiser_division_is_the_correctly_rounded_quotient():
    torch.cuda.init()
    d = tempfile.mkdtemp(prefix="qevict_div_")
    src = os.path.join(d, "div.cu")
    so = os.path.join(d, "libdiv.so")
    with open(src, "w") as f:
        f.write(_SRC)
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
                           "-Xcompiler", "-fPIC", f"-I{CSRC}", "-o", so, src])
    lib = ctypes.CDLL(so)
    bad = ctypes.c_ulonglong(0)
    first = (ctypes.c_float * 4)()
    rc = lib.run_div_check(ctypes.byref(bad), first)
    assert rc == 0, rc
    assert bad.value == 0, f"{bad.value} quotients differ; first: a={first[0]!r} b={first[1]!r} " \
                           f"got {first[2]!r}, correctly rounded {first[3]!r}"
