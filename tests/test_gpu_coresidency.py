"""The decode's splits wait for one another's records, so all CTAs of a
decode must be resident at once. These tests run a decode beside a kernel that
holds all SMs but ten for about 50 ms, with the inter-CTA wait limit cut to
about 1 ms: the cooperative grid (the default) starts when it fits and meets;
a non-cooperative grid strands the splits that fit, whose waits run out and
report TIMEOUT. A third test makes the waits run out on purpose (a limit of
one cycle). Each checks that nothing hangs and that after the status is
cleared the cache decodes as before. Nothing here faults or hangs a GPU: the
holding kernel sleeps on its own clock for a fixed time, and every wait of the
decode is bounded."""
import ctypes
import os
import subprocess
import tempfile
import time

import pytest
import torch

from tiered_kv_cache_decode_gb300 import synth
from parity_util import close, make_pair

pytestmark = pytest.mark.gpu

_HOLD_SRC = r"""
#include <cuda_runtime.h>
// Holds the SM it runs on: one CTA with most of the shared memory, whose
// first thread counts itself in (host-mapped counter), then sleeps in short
// steps until its own clock has advanced by `cycles` (a fixed, bounded time).
__global__ void hold_kernel(long long cycles, int *resident) {
    extern __shared__ char smem[];
    if (threadIdx.x == 0) {
        smem[0] = 1;
        atomicAdd_system(resident, 1);
        __threadfence_system();
        const long long t0 = clock64();
        while (clock64() - t0 < cycles) __nanosleep(2000);
    }
}
static int *g_host = nullptr, *g_dev = nullptr;
extern "C" int *hold_counter() {
    if (!g_host) {
        if (cudaHostAlloc((void **)&g_host, sizeof(int), cudaHostAllocMapped) != cudaSuccess) return nullptr;
        if (cudaHostGetDevicePointer((void **)&g_dev, g_host, 0) != cudaSuccess) return nullptr;
    }
    return g_host;
}
extern "C" int hold_sms(int ctas, long long cycles, int smem, void *stream) {
    if (!hold_counter()) return -1;
    *(volatile int *)g_host = 0;
    cudaError_t e = cudaFuncSetAttribute(hold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return (int)e;
    hold_kernel<<<ctas, 32, smem, (cudaStream_t)stream>>>(cycles, g_dev);
    return (int)cudaGetLastError();
}
"""

_hold = None


def _hold_lib():
    global _hold
    if _hold is None:
        d = tempfile.mkdtemp(prefix="qevict_hold_")
        src = os.path.join(d, "hold.cu")
        so = os.path.join(d, "libhold.so")
        with open(src, "w") as f:
            f.write(_HOLD_SRC)
        subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared",
                               "-Xcompiler", "-fPIC", "-o", so, src])
        _hold = ctypes.CDLL(so)
        _hold.hold_sms.argtypes = [ctypes.c_int, ctypes.c_longlong, ctypes.c_int, ctypes.c_void_p]
        _hold.hold_sms.restype = ctypes.c_int
        _hold.hold_counter.restype = ctypes.POINTER(ctypes.c_int)
    return _hold


HOLD_CYCLES = 100_000_000   # about 50 ms at GB300 clocks


def _hold_most(stream):
    """Start the holding kernel on all SMs but ten and return once all of its
    CTAs are resident (or after 2 s, which fails the test). The decode's CTAs
    go out in block order, so the ten that fit beside it are splits of one
    (sequence, KV head) whose other splits cannot start."""
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    hold = _hold_lib()
    ctas = n_sms - 10
    rc = hold.hold_sms(ctas, HOLD_CYCLES, 200 * 1024, ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0, rc
    cnt = hold.hold_counter()
    t_end = time.perf_counter() + 2.0
    while cnt[0] < ctas and time.perf_counter() < t_end:
        time.sleep(0.0002)
    assert cnt[0] == ctas, cnt[0]


def _decode_case():
    B, Hq, Hkv, w, L = 1, 32, 8, 64, 8192
    W = L // w
    scores = [synth.zipf_scores(0, 0, B, W)]
    cache, refs = make_pair(B, Hq, Hkv, w, L, beta=0.2, rho=0.5, scores=scores)
    q = synth.queries(0, 0, 0, B, Hq, 128)
    return cache, refs[0], q


def _warm(cache, q):
    """Device copies of the inputs and outputs, made before the holding kernel
    starts (an allocation while it runs could wait for it), and one decode, so
    that nothing in the timed call sets anything up."""
    qd = q.cuda()
    out = torch.empty(cache.B, cache.Hq, 128, dtype=torch.float32, device="cuda")
    mass = torch.empty(cache.B, cache.Hq, cache.num_windows(0), dtype=torch.float32, device="cuda")
    cache.decode(0, qd, out=out, mass=mass, accumulate=False)
    torch.cuda.synchronize()
    assert cache.status() == 0, cache.last_error()
    return qd, out, mass


def test_cooperative_decode_waits_for_sms_held_by_another_kernel():
    """The decode is launched while another kernel holds all SMs but ten for
    about 50 ms, with the inter-CTA wait limit cut to about 1 ms. The
    cooperative grid starts only when all of its CTAs fit, so no split waits
    for a CTA that is not resident: the status stays OK and the output is the
    oracle's."""
    cache, ref, q = _decode_case()
    ro, rm = ref.decode(q.float().numpy(), accumulate=False)
    qd, out, mass = _warm(cache, q)
    cache.set_wait_limit(2_000_000)
    s_hold, s_dec = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    _hold_most(s_hold)
    cache.decode(0, qd, out=out, mass=mass, accumulate=False, stream=s_dec)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert cache.status() == 0, cache.last_error()
    close(out.cpu().numpy(), ro, "attention output beside the holding kernel")
    close(mass.cpu().numpy(), rm, "window mass beside the holding kernel")
    assert 0.03 < elapsed < 1.0, elapsed   # it waited for the held SMs, not for its limit
    cache.set_wait_limit(0)


def test_non_cooperative_decode_beside_held_sms_reports_timeout_and_recovers():
    """The same, launched non-cooperatively: ten splits are resident and wait
    for the others of their (sequence, KV head), which the holding kernel keeps
    out for 50 ms.
    Their waits run out after about 1 ms and report TIMEOUT (no hang); after
    the status is cleared the cache decodes as before."""
    cache, ref, q = _decode_case()
    ro, rm = ref.decode(q.float().numpy(), accumulate=False)
    cache.set_cooperative_launch(False)
    qd, out, mass = _warm(cache, q)
    cache.set_wait_limit(2_000_000)
    s_hold, s_dec = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    _hold_most(s_hold)
    cache.decode(0, qd, out=out, mass=mass, accumulate=False, stream=s_dec)
    torch.cuda.synchronize()
    assert binding_status_name(cache.status()) == "TIMEOUT"
    cache.set_wait_limit(0)
    cache.clear_status()
    out, mass = cache.decode(0, q.cuda(), accumulate=False)
    torch.cuda.synchronize()
    assert cache.status() == 0, cache.last_error()
    close(out.cpu().numpy(), ro, "attention output after the timeout")
    close(mass.cpu().numpy(), rm, "window mass after the timeout")


def test_a_wait_that_runs_out_reports_timeout_and_the_cache_recovers():
    cache, ref, q = _decode_case()
    ro, rm = ref.decode(q.float().numpy(), accumulate=False)
    cache.set_wait_limit(1)
    cache.decode(0, q.cuda(), accumulate=False)
    torch.cuda.synchronize()
    assert binding_status_name(cache.status()) == "TIMEOUT"
    cache.set_wait_limit(0)
    cache.clear_status()
    for _ in range(2):
        out, mass = cache.decode(0, q.cuda(), accumulate=False)
        torch.cuda.synchronize()
        assert cache.status() == 0, cache.last_error()
        close(out.cpu().numpy(), ro, "attention output after the timeout")
        close(mass.cpu().numpy(), rm, "window mass after the timeout")


def binding_status_name(code):
    from tiered_kv_cache_decode_gb300 import binding
    return binding.STATUS.get(code, code)
