// Measurement-only diagnostics of the tiered cache: future missed mass.
//
// QEvict ("Technische Samenvatting: QEvict", Kernbijdragen) characterises a
// policy by the share of future attention that lands on states it has already
// discarded. Given the full keys of a layer (as they were before any tier
// move; the caller keeps them for the measurement) and a query, this computes
// dense softmax attention over all tokens and sums the probability of the
// tokens whose window the cache has evicted.
#include "qevict_internal.cuh"

#include <math.h>

namespace qevict {
namespace {

constexpr int kFmmWarps = 8;
constexpr float kLog2eF = 1.4426950408889634f;

// (max, sum of 2^(x - max) over all tokens, the same over evicted tokens)
struct FmmStat {
    float m, la, le;
};

__device__ __forceinline__ FmmStat fmm_merge(FmmStat a, FmmStat b) {
    if (b.m == -INFINITY) return a;
    if (a.m == -INFINITY) return b;
    const float m = fmaxf(a.m, b.m);
    const float fa = exp2f(a.m - m), fb = exp2f(b.m - m);
    return FmmStat{m, a.la * fa + b.la * fb, a.le * fa + b.le * fb};
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint4 &a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr long long kFmmWaitCycles = 4000000000ll;   // about two seconds at GB300 clocks

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// suspends the thread until the phase completes or about 20 us pass
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}
// bounded wait: false after about two seconds
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kFmmWaitCycles) return false;
    return true;
}
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z, uint32_t bar,
                                       uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint4 &r) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr));
}

// Running (max, sums) of one head over two more logits (log2 domain).
__device__ __forceinline__ void fmm_add2(FmmStat &st, float x0, float x1, bool ok0, bool ok1, bool evicted) {
    x0 = ok0 ? x0 : -INFINITY;
    x1 = ok1 ? x1 : -INFINITY;
    const float m = fmaxf(st.m, fmaxf(x0, x1));
    if (m == -INFINITY) return;
    const float f = ex2(st.m - m), e = ex2(x0 - m) + ex2(x1 - m);
    st.la = fmaf(st.la, f, e);
    st.le = st.le * f + (evicted ? e : 0.f);
    st.m = m;
}

// Each warp streams chunks of 16 tokens through its own ring of kFmmStages
// stages in shared memory. A stage holds the chunk's keys as two TMA boxes of
// 16 tokens x 64 channels (channels 0-63, then 64-127), 128-byte rows with
// the 128-byte swizzle, so that ldmatrix reads them without bank conflicts.
constexpr int kFmmStages = 3;
constexpr int kFmmThreads = kFmmWarps * 32;
constexpr int kFmmStage = 4096;
constexpr int kFmmRing = kFmmWarps * kFmmStages * kFmmStage;
constexpr int kFmmSmem = kFmmRing + kFmmWarps * kFmmStages * 8 + 1024;   // + barriers, + alignment

// One CTA per (split of the token range, sequence and KV head), two CTAs per
// SM (one's first chunks and merge overlap the other's streaming); splits
// start on 16-token boundaries, so a chunk of 16 tokens lies
// inside one window (a window is a multiple of 16 tokens) and takes one tier
// byte. A warp takes every 8th chunk: lane 0 issues the chunk's two TMA
// copies kFmmStages - 1 chunks ahead, and the warp computes the logits on the
// tensor cores (mma.sync m16n8k16, bf16 operands, fp32 sums) with the tokens
// as the M rows (A from ldmatrix), the query heads of the group as the N
// columns (padded to 8) and the channels as K in 8 steps of 16. Lane
// (g, c) = (lane / 4, lane % 4) keeps a running (max, sums) for heads 2c and
// 2c + 1.
//
// The CTA's statistics per head go to `part`; the last CTA of each (sequence,
// KV head) to arrive on `cnt` (zero between launches, reset by that CTA)
// merges all splits and writes the missed mass of the group's heads.
template <int G>
__global__ void __launch_bounds__(kFmmThreads, 2) fmm_kernel(const LayerDev D, const CacheDev C,
                                                             const __grid_constant__ CUtensorMap kmap, int layer,
                                                             const __nv_bfloat16 *q, int L, float *part,
                                                             int splits, uint32_t *cnt, float *fmm) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int split = blockIdx.x, bk = blockIdx.y;
    const int b = bk / D.Hkv, kvh = bk % D.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, c = lane & 3;
    const float scale = kLog2eF * rsqrtf((float)kHeadDim);
    const uint32_t sraw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t ring = (sraw + 1023u) & ~1023u;   // swizzled TMA boxes want 1024-byte alignment
    const uint32_t wring = ring + warp * kFmmStages * kFmmStage;
    const uint32_t bars = ring + kFmmRing + warp * kFmmStages * 8;

    const int nch = (L + 15) / 16;
    const int t0 = 16 * (int)((int64_t)nch * split / splits);
    const int t1 = min(L, 16 * (int)((int64_t)nch * (split + 1) / splits));
    const uint8_t *tier = D.tier + (int64_t)b * D.Wmax;
    auto chunk0 = [&](int k) { return t0 + (warp + k * kFmmWarps) * 16; };
    // the unit's KV head and first token in the map (a unit may be a (sequence, KV head) pair)
    const int ky = (b % D.hs) * D.Hkv + kvh, kz = (b / D.hs) * L;

    if (lane == 0)
        for (int i = 0; i < kFmmStages; ++i) mbar_init(bars + 8 * i, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncwarp();
    const uint64_t pol = evict_first_policy();
    auto issue = [&](int k) {   // lane 0
        const int st = k % kFmmStages, c0 = chunk0(k);
        const uint32_t bar = bars + 8 * st, dst = wring + st * kFmmStage;
        mbar_expect_tx(bar, (uint32_t)kFmmStage);
        tma_3d(dst, &kmap, 0, ky, kz + c0, bar, pol);
        tma_3d(dst + 2048, &kmap, 64, ky, kz + c0, bar, pol);
    };
    int issued = 0;
    if (lane == 0)
        for (; issued < kFmmStages - 1 && chunk0(issued) < t1; ++issued) issue(issued);
    issued = __shfl_sync(0xffffffffu, issued, 0);

    // B fragments (q^T): step ks, (k = 2c, 2c+1) and (k = 2c+8, 2c+9) of head g
    uint32_t qb[8][2];
    {
        const uint32_t *qp = reinterpret_cast<const uint32_t *>(q + ((int64_t)b * D.Hq + kvh * G + g) * kHeadDim);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            qb[ks][0] = g < G ? qp[8 * ks + c] : 0u;
            qb[ks][1] = g < G ? qp[8 * ks + 4 + c] : 0u;
        }
    }
    FmmStat st[2] = {{-INFINITY, 0.f, 0.f}, {-INFINITY, 0.f, 0.f}};
    // ldmatrix row of this lane: matrix m = lane / 8 gives tokens 0-7 or 8-15 and k 0-7 or 8-15
    const int lm_tok = (lane & 7) + 8 * ((lane >> 3) & 1), lm_hi = lane >> 4;

    for (int k = 0; k < issued; ++k) {
        const int sidx = k % kFmmStages, c0 = chunk0(k);
        const bool ev = tier[c0 / D.w] == QEVICT_TIER_E;
        const bool ok = mbar_wait(bars + 8 * sidx, (uint32_t)((k / kFmmStages) & 1));
        if (__any_sync(0xffffffffu, !ok)) {
            if (lane == 0) {
                set_status(C, QEVICT_ERR_TIMEOUT, layer, b, -5);
                // the copies still in flight land before the CTA leaves
                for (int r = k; r < issued; ++r)
                    (void)mbar_wait(bars + 8 * (r % kFmmStages), (uint32_t)((r / kFmmStages) & 1));
            }
            break;
        }
        const uint32_t base = wring + sidx * kFmmStage;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int chunk = 2 * (ks & 3) + lm_hi;
            uint4 a;
            ldsm_x4(base + (ks >> 2) * 2048 + lm_tok * 128 + ((chunk ^ (lm_tok & 7)) << 4), a);
            mma_bf16(acc, a, qb[ks][0], qb[ks][1]);
        }
        __syncwarp();   // every lane has read the stage before it is refilled
        if (lane == 0 && chunk0(issued) < t1) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(issued);
        }
        issued = (chunk0(issued) < t1) ? issued + 1 : issued;
        // acc: (token g, head 2c), (token g, head 2c+1), (token g+8, head 2c), (token g+8, head 2c+1)
        const bool ok0 = c0 + g < t1, ok1 = c0 + g + 8 < t1;
        if (2 * c < G) fmm_add2(st[0], acc[0] * scale, acc[2] * scale, ok0, ok1, ev);
        if (2 * c + 1 < G) fmm_add2(st[1], acc[1] * scale, acc[3] * scale, ok0, ok1, ev);
    }

    // per head: merge the 8 lanes that share c, then the warps
    __shared__ FmmStat s_st[kFmmWarps][8];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        FmmStat a = st[j];
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1) {
            const FmmStat p{__shfl_xor_sync(0xffffffffu, a.m, o), __shfl_xor_sync(0xffffffffu, a.la, o),
                            __shfl_xor_sync(0xffffffffu, a.le, o)};
            a = fmm_merge(a, p);
        }
        if (g == 0) s_st[warp][2 * c + j] = a;
    }
    __syncthreads();
    if (threadIdx.x < G) {
        FmmStat acc{-INFINITY, 0.f, 0.f};
        for (int w = 0; w < kFmmWarps; ++w) acc = fmm_merge(acc, s_st[w][threadIdx.x]);
        float *o = part + (((int64_t)bk * splits + split) * G + threadIdx.x) * 3;
        o[0] = acc.m;
        o[1] = acc.la;
        o[2] = acc.le;
        __threadfence();
    }
    __shared__ bool s_last;
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&cnt[2 * bk], 1u) == (unsigned)splits - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // warp hh merges head hh over the splits, lanes taking splits in turn
    if (warp < G) {
        FmmStat a{-INFINITY, 0.f, 0.f};
        for (int sp = lane; sp < splits; sp += 32) {
            const float *o = part + (((int64_t)bk * splits + sp) * G + warp) * 3;
            a = fmm_merge(a, FmmStat{__ldcg(o), __ldcg(o + 1), __ldcg(o + 2)});
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const FmmStat p{__shfl_xor_sync(0xffffffffu, a.m, o), __shfl_xor_sync(0xffffffffu, a.la, o),
                            __shfl_xor_sync(0xffffffffu, a.le, o)};
            a = fmm_merge(a, p);
        }
        if (lane == 0) fmm[(int64_t)b * D.Hq + kvh * G + warp] = a.la > 0.f ? a.le / a.la : 0.f;
    }
    if (threadIdx.x == 0) cnt[2 * bk] = 0;
}

}  // namespace

cudaError_t launch_future_missed_mass(const LayerDev &L, const CacheDev &C, const DecodeScratch &S, int layer,
                                      const CUtensorMap &kmap, const __nv_bfloat16 *q, int n_tokens, float *fmm,
                                      int num_sms, cudaStream_t s) {
    const int pairs = L.B * L.Hkv;
    // Partials (3 floats per split and query head) go to the window-statistics
    // area of the decode scratch, which holds 8 Wmax bytes (at least 12) per
    // query head and carries nothing from one decode launch to the next. (The
    // partial output area is not used: its words carry arrival tags.)
    float *part = reinterpret_cast<float *>(S.wstat);
    // The split arrival counters of the decode scratch (zero between launches)
    // count this launch's arrivals too; every launch leaves them at zero.
    uint32_t *cnt = S.bar;   // [B*Hkv][2]; the kernel counts on entry 2 * bk
    // two CTAs per SM, spread over the (sequence, KV head) pairs
    auto grid_for = [&](const void *fn) {
        const cudaError_t e = once_per_device(L.G, [fn]() {
            return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kFmmSmem);
        });
        if (e != cudaSuccess) return -1;
        const int splits = (2 * num_sms + pairs - 1) / pairs;
        return max(1, min(splits, min(256, 2 * L.Wmax / 3)));
    };
    switch (L.G) {
#define QV_CASE(GG)                                                                                          \
    case GG: {                                                                                               \
        const int splits = grid_for((const void *)fmm_kernel<GG>);                                           \
        if (splits < 0) return cudaGetLastError();                                                           \
        fmm_kernel<GG><<<dim3(splits, pairs), kFmmThreads, kFmmSmem, s>>>(L, C, kmap, layer, q, n_tokens,    \
                                                                           part, splits, cnt, fmm);          \
        break;                                                                                               \
    }
        QV_CASE(1)
        QV_CASE(2)
        QV_CASE(3)
        QV_CASE(4)
        QV_CASE(5)
        QV_CASE(6)
        QV_CASE(7)
        QV_CASE(8)
#undef QV_CASE
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace qevict
