// Cache management kernels: layer initialisation, appends, the tier plan
// (routing, explicit tiers, prefill, listed demotions / promotions), the
// INT2 quantiser, the promotion dequantiser and the score reduction.
//
// Method: "Technische Samenvatting: QEvict" (gist.science 2608.05326),
// "Methodologie: QEvict" and "Kernmechanismen" (window routing under a byte
// budget, cumulative scoring, demotion, promotion, write-once ledger).
#include "qevict_internal.cuh"
#include "qevict_div.cuh"

#include <cooperative_groups.h>
namespace cg = cooperative_groups;

#include <math.h>

namespace qevict {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPlanMaxW = 4096;

// ---------------------------------------------------------------- init
__global__ void init_layer_kernel(LayerDev D) {
    const int64_t nW = (int64_t)D.B * D.Wmax;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int64_t i = i0; i < nW; i += stride) {
        D.tier[i] = QEVICT_TIER_E;
        D.fp_slot[i] = -1;
        D.lg_slot[i] = -1;
        D.lwrites[i] = 0;
        D.lbits[i] = 0;
    }
    for (int64_t i = i0; i < nW * D.Hkv; i += stride) D.score_part[i] = 0.f;
    for (int64_t i = i0; i < (int64_t)D.B * D.CF; i += stride) {
        const int b = (int)(i / D.CF), j = (int)(i % D.CF);
        D.fp_free[i] = b * D.CF + (D.CF - 1 - j);   // top of the stack pops slot b*CF first
    }
    for (int64_t i = i0; i < (int64_t)D.B * D.CQ; i += stride) {
        const int b = (int)(i / D.CQ), j = (int)(i % D.CQ);
        D.lg_free[i] = b * D.CQ + (D.CQ - 1 - j);
    }
    for (int64_t i = i0; i < D.B; i += stride) {
        int32_t *c = D.ctr + i * kCtrN;
        for (int k = 0; k < kCtrN; ++k) c[k] = 0;
        c[CTR_NEXT] = (int)i * D.CF;      // slot b*CF, the top of the stack, is taken ahead
        c[CTR_FP_TOP] = D.CF - 1;
        c[CTR_LG_TOP] = D.CQ;
    }
}

// ---------------------------------------------------------------- append
// One CTA per sequence: thread 0 opens the windows that start inside the
// appended range (a slot from the free list each), then the CTA copies the
// tokens' K and V rows into their windows' full-precision slots.
__global__ void append_kernel(LayerDev D, CacheDev C, int layer, const __nv_bfloat16 *__restrict__ k,
                              const __nv_bfloat16 *__restrict__ v, int n_new) {
    const int b = blockIdx.x;
    const int w = D.w;
    const int64_t wb = (int64_t)b * D.Wmax;
    __shared__ int s_bad;
    __shared__ int s_len;
    if (threadIdx.x == 0) {
        s_bad = 0;
        int32_t *ctr = D.ctr + b * kCtrN;
        const int64_t L0 = ctr[CTR_LEN];
        s_len = (int)L0;
        if (L0 + n_new > D.max_context) {
            set_status(C, QEVICT_ERR_INVALID_ARG, layer, b, (int)L0);
            s_bad = 1;
        } else if (L0 % w != 0) {
            const int wi = (int)(L0 / w);
            if (D.tier[wb + wi] != QEVICT_TIER_FP || D.fp_slot[wb + wi] < 0) {
                set_status(C, QEVICT_ERR_STATE, layer, b, wi);
                s_bad = 1;
            }
        }
        if (!s_bad) {
            for (int64_t p = ((L0 + w - 1) / w) * w; p < L0 + n_new; p += w) {
                const int wi = (int)(p / w);
                const int slot = ctr[CTR_NEXT];
                const int top = ctr[CTR_FP_TOP];
                if (top > 0) {
                    ctr[CTR_NEXT] = D.fp_free[b * D.CF + top - 1];
                    ctr[CTR_FP_TOP] = top - 1;
                } else {
                    ctr[CTR_NEXT] = -1;
                }
                if (slot < 0) set_status(C, QEVICT_ERR_CAPACITY, layer, b, wi);
                D.tier[wb + wi] = slot >= 0 ? QEVICT_TIER_FP : QEVICT_TIER_E;
                D.fp_slot[wb + wi] = slot;
                D.lg_slot[wb + wi] = -1;
                D.lwrites[wb + wi] = 0;
                for (int h = 0; h < D.Hkv; ++h) D.score_part[((int64_t)b * D.Hkv + h) * D.Wmax + wi] = 0.f;
                if (slot >= 0) {
                    const int n = ctr[CTR_NFP];
                    D.fp_list[b * D.CF + n] = make_int2(wi, slot);
                    ctr[CTR_NFP] = n + 1;
                }
            }
            ctr[CTR_LEN] = (int)(L0 + n_new);
        }
    }
    __syncthreads();
    if (s_bad) return;
    const int64_t L0 = s_len;
    constexpr int kChunks = kHeadDim * 2 / 16;   // 16-byte chunks per row
    const int64_t total = (int64_t)n_new * D.Hkv * 2 * kChunks;
    for (int64_t i = threadIdx.x; i < total; i += blockDim.x) {
        const int c = (int)(i % kChunks);
        int64_t r = i / kChunks;
        const int kv = (int)(r % 2);
        r /= 2;
        const int h = (int)(r % D.Hkv);
        const int t = (int)(r / D.Hkv);
        const int64_t p = L0 + t;
        const int wi = (int)(p / w), row = (int)(p % w);
        const int slot = D.fp_slot[wb + wi];
        if (slot < 0) continue;
        const __nv_bfloat16 *src = (kv ? v : k) + src_row(D, b, n_new, t, h) * kHeadDim;
        __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(D.fp_pool + (int64_t)slot * D.fp_slot_bytes) +
                             fp_off(h, kv, w, row, 8 * c);
        *reinterpret_cast<uint4 *>(dst) = reinterpret_cast<const uint4 *>(src)[c];
    }
}

// ---------------------------------------------------------------- plan
// Take a free full-precision slot ahead of time for the next window to open.
__device__ __forceinline__ void reserve_next(const LayerDev &D, int32_t *ctr, int b) {
    if (ctr[CTR_NEXT] < 0 && ctr[CTR_FP_TOP] > 0) {
        const int top = ctr[CTR_FP_TOP] - 1;
        ctr[CTR_NEXT] = D.fp_free[b * D.CF + top];
        ctr[CTR_FP_TOP] = top;
    }
}

__device__ __forceinline__ uint32_t orderable(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Rank of a window `age` windows before the open one under the log-sparse
// positional order, lowest first: (round, region, age) packed into 24 bits.
// The `recent` newest windows are dense (round 0); region l >= 1 covers ages
// [recent 2^(l-1), recent 2^l) and its offset m joins in round
// 1 + l - min(l, trailing zeros of m) (m = 0 counts as l trailing zeros):
// spacing 2^l in round 1, half of it in each later round.
__device__ __forceinline__ uint32_t logsparse_rank(int age, int recent) {
    if (age < recent) return (uint32_t)age;
    int region = 1;
    while (age >= (recent << region)) ++region;
    const int m = age - (recent << (region - 1));
    const int tz = m == 0 ? region : min(region, __ffs(m) - 1);
    return ((uint32_t)(1 + region - tz) << 20) | ((uint32_t)region << 12) | (uint32_t)age;
}

// Exclusive prefix sum over the block of one int per thread; *total gets the sum.
// N exclusive prefix sums over the block at once (three barriers in all):
// excl[n] is the sum of v[n] over the threads before this one, tot[n] over all.
// s_warp holds N * (kPlanThreads / 32) ints.
template <int N>
__device__ void block_scan_n(const int (&v)[N], int (&excl)[N], int (&tot)[N], int *s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int nwarp = kPlanThreads / 32;
    int x[N];
#pragma unroll
    for (int n = 0; n < N; ++n) {
        x[n] = v[n];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x[n], o);
            if (lane >= o) x[n] += y;
        }
        if (lane == 31) s_warp[n * nwarp + warp] = x[n];
    }
    __syncthreads();
    if (warp < N) {
        int ws = s_warp[warp * nwarp + lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, ws, o);
            if (lane >= o) ws += y;
        }
        s_warp[warp * nwarp + lane] = ws;
    }
    __syncthreads();
#pragma unroll
    for (int n = 0; n < N; ++n) {
        excl[n] = x[n] - v[n] + (warp > 0 ? s_warp[n * nwarp + warp - 1] : 0);
        tot[n] = s_warp[n * nwarp + nwarp - 1];
    }
    __syncthreads();
}

__device__ int block_scan(int v, int *total, int *s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int nwarp = kPlanThreads / 32;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int ws = lane < nwarp ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, ws, o);
            if (lane >= o) ws += y;
        }
        if (lane < nwarp) s_warp[lane] = ws;
    }
    __syncthreads();
    const int excl = x - v + (warp > 0 ? s_warp[warp - 1] : 0);
    *total = s_warp[nwarp - 1];
    __syncthreads();
    return excl;
}

// Score of a routing sort key (the float behind ~orderable(S) in the high word).
__device__ __forceinline__ double key_score(unsigned long long key) {
    const uint32_t o = ~(uint32_t)(key >> 32);
    const uint32_t u = (o & 0x80000000u) ? (o & 0x7fffffffu) : ~o;
    return (double)__uint_as_float(u);
}

// ---------------------------------------------------------------- mixed widths
// Rate-distortion allocation over widths {0, 2, 4, 8, 16} ("Technische
// Samenvatting: RDKV", 2.1-2.2, the Lagrangian of the multiple-choice
// knapsack). A window's options form a chain of widths: 0, 2, 4, 8, 16 (those
// the ledger can hold) for a window never quantised, 0, b, 16 for one whose
// ledger entry has width b. Each chain step a -> b is an upgrade with gain
// (2^-a - 2^-b) / (cost(b) - cost(a)) * s per byte (float64), s the window's
// score; upgrades are taken by gain, highest first (lower step, then rank, on
// a tie), while positive, until the first that does not fit.
constexpr int kMixClasses = 4;    // never quantised; ledger width 2, 4, 8
constexpr int kMixTypes = 10;     // (class, step) lists: 4 + 2 + 2 + 2

__device__ __forceinline__ int mix_steps(int ci, int maxP) {
    return ci == 0 ? 2 + (maxP >= 2) + (maxP >= 4) : 2;
}
__device__ __forceinline__ int mix_width(int ci, int idx, int maxP) {
    if (idx == 0) return 0;
    if (ci != 0) return idx == 1 ? (2 << (ci - 1)) : 16;
    return idx < mix_steps(0, maxP) ? (2 << (idx - 1)) : 16;
}
__device__ __forceinline__ int64_t mix_cost(const LayerDev &D, int bits) {
    if (bits == 0) return 0;
    if (bits == 16) return D.c_fp;
    return (int64_t)D.w * D.Hkv * 2 * (kHeadDim * bits / 8 + 4 * kGroups);
}
__device__ __forceinline__ double exp2_neg(int a) {   // 2^-a, exact
    return __longlong_as_double((long long)(1023 - a) << 52);
}
__device__ __forceinline__ unsigned long long orderable64(double x) {
    const unsigned long long u = (unsigned long long)__double_as_longlong(x);
    return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}
__device__ __forceinline__ int mix_class(int lbits) { return lbits == 0 ? 0 : lbits == 2 ? 1 : lbits == 4 ? 2 : 3; }

// Target tiers of the ranked candidates (s_key[0] the open window, s_key[1 +
// j] the rest in rank order). The taken upgrades are a prefix of the global
// order, and along each (class, step) list of windows in rank order the gain
// does not rise, so an upgrade is taken iff its gain is positive and the cost
// of the prefix through it fits; that prefix is counted by a binary search in
// every list. dyn: [upgrades] orderable gains, then [n] rank indices grouped
// by class.
__device__ void rd_mixed_targets(const LayerDev &D, const unsigned long long *s_key, uint8_t *s_tgt, int ncand,
                                 int64_t budget, int64_t wb, int *s_warp, unsigned long long *dyn) {
    __shared__ int s_coff[kMixClasses + 1], s_toff[kMixTypes + 1], s_tfirst[kMixClasses], s_take[kMixTypes];
    __shared__ int s_tcls[kMixTypes], s_tstep[kMixTypes], s_ntypes;
    __shared__ double s_tk[kMixTypes];
    __shared__ long long s_tcost[kMixTypes];
    const int tid = threadIdx.x, n = ncand - 1, maxP = D.maxP;
    if (tid == 0 && ncand > 0) s_tgt[(int)(s_key[0] & 0xffffffffu)] = QEVICT_TIER_FP;   // no candidate: key 0 is unset
    if (n <= 0) {
        __syncthreads();
        return;
    }
    // ---- group the rest by class, rank order kept within a class
    const int per = (n + kPlanThreads - 1) / kPlanThreads;
    const int j0 = tid * per, j1 = min(n, j0 + per);
    int cnt[kMixClasses] = {0, 0, 0, 0};
    for (int j = j0; j < j1; ++j) ++cnt[mix_class(D.lbits[wb + (int)(s_key[1 + j] & 0xffffffffu)])];
    int excl[kMixClasses], tot[kMixClasses];
#pragma unroll
    for (int c = 0; c < kMixClasses; ++c) excl[c] = block_scan(cnt[c], &tot[c], s_warp);
    uint16_t *s_rk = reinterpret_cast<uint16_t *>(dyn + (size_t)mix_steps(0, maxP) * D.Wmax);
    if (tid == 0) {
        int off = 0, t = 0;
        for (int c = 0; c < kMixClasses; ++c) {
            s_coff[c] = off;
            off += tot[c];
        }
        s_coff[kMixClasses] = off;
        int toff = 0;
        for (int c = 0; c < kMixClasses; ++c) {
            s_tfirst[c] = t;
            for (int i = 0; i < mix_steps(c, maxP); ++i, ++t) {
                const int a = mix_width(c, i, maxP), bw = mix_width(c, i + 1, maxP);
                const int64_t cost = mix_cost(D, bw) - mix_cost(D, a);
                s_tk[t] = (exp2_neg(a) - exp2_neg(bw)) / (double)cost;
                s_tcost[t] = cost;
                s_tcls[t] = c;
                s_tstep[t] = i;
                s_toff[t] = toff;
                s_take[t] = 0;
                toff += tot[c];
            }
        }
        s_toff[t] = toff;
        s_ntypes = t;
    }
    __syncthreads();
    {
        int run[kMixClasses] = {0, 0, 0, 0};
        for (int j = j0; j < j1; ++j) {
            const int c = mix_class(D.lbits[wb + (int)(s_key[1 + j] & 0xffffffffu)]);
            s_rk[s_coff[c] + excl[c] + run[c]++] = (uint16_t)j;
        }
    }
    __syncthreads();
    const int nt = s_ntypes, U = s_toff[nt];
    // ---- one gain per upgrade, list by list
    for (int e = tid; e < U; e += kPlanThreads) {
        int t = 0;
        while (e >= s_toff[t + 1]) ++t;
        const int j = s_rk[s_coff[s_tcls[t]] + e - s_toff[t]];
        dyn[e] = orderable64(s_tk[t] * key_score(s_key[1 + j]));
    }
    __syncthreads();
    // ---- which upgrades are taken: positive gain and the prefix through it fits
    const int64_t room = budget - D.c_fp;
    for (int e = tid; e < U; e += kPlanThreads) {
        const unsigned long long g = dyn[e];
        if (g <= 0x8000000000000000ull) continue;   // gain <= 0
        int t = 0;
        while (e >= s_toff[t + 1]) ++t;
        const int step = s_tstep[t];
        const int j = s_rk[s_coff[s_tcls[t]] + e - s_toff[t]];
        int64_t prefix = s_tcost[t];
        for (int t2 = 0; t2 < nt && prefix <= room; ++t2) {
            const int base = s_toff[t2], len = s_toff[t2 + 1] - base, step2 = s_tstep[t2];
            const int cbase = s_coff[s_tcls[t2]];
            int lo = 0, hi = len;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                const unsigned long long g2 = dyn[base + mid];
                const bool before = g2 > g || (g2 == g && (step2 < step || (step2 == step && s_rk[cbase + mid] < j)));
                if (before)
                    lo = mid + 1;
                else
                    hi = mid;
            }
            prefix += (int64_t)lo * s_tcost[t2];
        }
        if (prefix <= room) atomicAdd(&s_take[t], 1);
    }
    __syncthreads();
    // ---- each window's width: the steps of its chain taken, in order
    {
        int run[kMixClasses] = {0, 0, 0, 0};
        for (int j = j0; j < j1; ++j) {
            const int wi = (int)(s_key[1 + j] & 0xffffffffu);
            const int c = mix_class(D.lbits[wb + wi]);
            const int q = excl[c] + run[c]++;
            int st = 0;
            while (st < mix_steps(c, maxP) && q < s_take[s_tfirst[c] + st]) ++st;
            const int bits = mix_width(c, st, maxP);
            s_tgt[wi] = bits == 16 ? QEVICT_TIER_FP
                        : bits == 8 ? QEVICT_TIER_Q8
                        : bits == 4 ? QEVICT_TIER_Q4
                        : bits == 2 ? QEVICT_TIER_Q
                                    : QEVICT_TIER_E;
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------------- K-channel widths
// "Technische Samenvatting: RDKV", 2.2 Fase 3: after the window widths, the
// 32-channel K groups of the sequence's KV heads (units (KV head, group))
// take widths along 0 -> 2 -> 4 -> 8 within the K bytes the quantised windows
// have at their widths. A group costs 4 b + 4 bytes per token; the step a -> b
// of a group of weight W (its channels' weights added in channel order,
// float64) gains (2^-a - 2^-b) / (tokens (cost(b) - cost(a))) * W per byte.
// Steps are taken by gain, highest first (lower step, then lower unit, on a
// tie), while positive, until the first that does not fit. Units are at most
// 64 (KV heads <= 16), steps at most 192.
constexpr int kKchMaxUnits = 64;
__device__ __forceinline__ int kgroup_cost(int bits) { return kGroup * bits / 8 + 4; }
__device__ void k_channel_widths(const LayerDev &D, const float *kweights, const uint8_t *s_tgt, int nw, int b,
                                 int *s_warp) {
    __shared__ double s_wg[kKchMaxUnits], s_gain[3 * kKchMaxUnits], s_kstep[3];
    __shared__ short s_ord[3 * kKchMaxUnits];
    __shared__ long long s_cost[3];
    const int tid = threadIdx.x, U = D.Hkv * kGroups, E = 3 * U;
    // quantised windows by width
    int c2 = 0, c4 = 0, c8 = 0;
    for (int i = tid; i < nw; i += kPlanThreads) {
        const uint8_t t = s_tgt[i];
        c2 += t == QEVICT_TIER_Q;
        c4 += t == QEVICT_TIER_Q4;
        c8 += t == QEVICT_TIER_Q8;
    }
    int cv[3] = {c2, c4, c8}, co[3], ct[3];
    block_scan_n<3>(cv, co, ct, s_warp);
    const int64_t n_tok = (int64_t)(ct[0] + ct[1] + ct[2]) * D.w;
    // K budget: the K halves of the quantised windows at their widths
    const int64_t kbud = (int64_t)D.w * D.Hkv *
                         ((int64_t)ct[0] * (16 * 2 + 16) + (int64_t)ct[1] * (16 * 4 + 16) + (int64_t)ct[2] * (16 * 8 + 16));
    if (tid < U) {
        const float *wp = kweights + ((int64_t)b * D.Hkv + tid / kGroups) * kHeadDim + (tid % kGroups) * kGroup;
        double W = 0.0;
        for (int c = 0; c < kGroup; ++c) W += (double)wp[c];
        s_wg[tid] = W;
    }
    if (tid < 3) {
        const int a0 = tid == 0 ? 0 : (2 << (tid - 1)), b0 = 2 << tid;
        const long long cost = (long long)n_tok * (kgroup_cost(b0) - kgroup_cost(a0));
        s_cost[tid] = cost;
        s_kstep[tid] = cost > 0 ? (exp2_neg(a0) - exp2_neg(b0)) / (double)cost : 0.0;
    }
    __syncthreads();
    // step e = (step i, unit u): its place in the order by (gain desc, step asc, unit asc)
    if (tid < E) s_gain[tid] = s_kstep[tid / U] * s_wg[tid % U];
    __syncthreads();
    if (tid < E) {
        const double g0 = s_gain[tid];
        const int i0 = tid / U, u0 = tid % U;
        int pos = 0;
        for (int e = 0; e < E; ++e) {
            const double g = s_gain[e];
            const int i = e / U, u = e % U;
            pos += g > g0 || (g == g0 && (i < i0 || (i == i0 && u < u0)));
        }
        s_ord[pos] = (short)tid;
    }
    __syncthreads();
    if (tid == 0) {
        int steps[kKchMaxUnits];
        for (int u = 0; u < U; ++u) steps[u] = 0;
        if (n_tok > 0) {
            long long used = (long long)n_tok * U * kgroup_cost(0);
            for (int r = 0; r < E; ++r) {
                const int e = s_ord[r], i = e / U, u = e % U;
                if (!(s_gain[e] > 0.0) || used + s_cost[i] > kbud) break;
                used += s_cost[i];
                steps[u] = i + 1;   // along a chain the gain falls, so a unit's steps come in order
            }
        }
        for (int u = 0; u < U; ++u) D.kgw[(int64_t)b * U + u] = (uint8_t)(steps[u] == 0 ? 0 : (2 << (steps[u] - 1)));
        D.ctr[b * kCtrN + CTR_KCH] = 1;
    }
    __syncthreads();
}

// One CTA per sequence. Computes the target tier of every window (by ranking
// the cumulative scores under the budget, or from explicit tiers), then
// applies the transitions: free the slots of evicted / demoted windows, take
// slots for promotions and first quantisations, update the window table,
// queue the data movement (quantise, dequantise, prefill copy) and rebuild
// the per-tier window lists the decode kernel walks.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(LayerDev D, CacheDev C, PlanArgs a) {
    __shared__ unsigned long long s_key[kPlanMaxW];
    __shared__ uint8_t s_cur[kPlanMaxW];
    __shared__ uint8_t s_tgt[kPlanMaxW];
    __shared__ uint8_t s_old[kPlanMaxW];   // tiers before this plan, for the move's counts
    __shared__ int s_warp[4 * (kPlanThreads / 32)];
    __shared__ int s_cnt[8];
    __shared__ long long s_budget;
    __shared__ int s_nfp_budget;
    extern __shared__ unsigned long long s_dyn[];   // the mixed-width route's gains and lists

    const int b = blockIdx.x, tid = threadIdx.x;
    const int64_t wb = (int64_t)b * D.Wmax;
    int32_t *ctr = D.ctr + b * kCtrN;
    const bool prefill = a.mode == PLAN_PREFILL_SCORES || a.mode == PLAN_PREFILL_TIERS;
    const int64_t length = prefill ? a.prefill_len : (int64_t)ctr[CTR_LEN];
    const int nw = (int)((length + D.w - 1) / D.w);
    const bool partial_last = (length % D.w) != 0;
    if (tid < 8) s_cnt[tid] = 0;
    // the tiers as they are (loaded before thread 0's counter updates, which do not touch them)
    for (int i = tid; i < nw; i += kPlanThreads) s_old[i] = s_cur[i] = prefill ? QEVICT_TIER_FP : D.tier[wb + i];
    if (tid == 0) {   // nothing queued unless this plan queues it
        ctr[CTR_WQ] = 0;
        ctr[CTR_WP] = 0;
        ctr[CTR_WC] = 0;
        // the slot reserved for the next window goes back on the free list for the plan
        const int nx = ctr[CTR_NEXT];
        if (nx >= 0) {
            D.fp_free[b * D.CF + ctr[CTR_FP_TOP]] = nx;
            ctr[CTR_FP_TOP] += 1;
            ctr[CTR_NEXT] = -1;
        }
    }
    __syncthreads();
    if (nw == 0) {
        if (tid == 0) reserve_next(D, ctr, b);
        return;
    }
    // byte budget at this length: B_t = floor(beta * L * Hkv * d * 4), and the full-precision
    // count of the share rule (float64, once, by thread 0: the double division is slow)
    if (tid == 0) {
        const int64_t bt = (int64_t)floor(D.beta * (double)(length * D.Hkv * kHeadDim * 4));
        s_budget = bt;
        s_nfp_budget = (int)floor((D.rho * (double)bt) / (double)D.c_fp);
    }
    __syncthreads();
    const int64_t budget = s_budget;
    const int nfp_budget = s_nfp_budget;
    if ((a.mode == PLAN_ROUTE || a.mode == PLAN_PREFILL_SCORES || a.mode == PLAN_LOGSPARSE || a.mode == PLAN_RD ||
         a.mode == PLAN_RD_MIXED || a.mode == PLAN_RD_KV) &&
        budget < D.c_fp) {
        if (tid == 0) {
            set_status(C, QEVICT_ERR_BUDGET, a.layer, b, (int)length);
            reserve_next(D, ctr, b);
        }
        return;
    }

    if (a.mode == PLAN_DEMOTE || a.mode == PLAN_PROMOTE) {
        // Listed transitions, applied one by one in list order.
        if (tid == 0) {
            int nq = 0, np = 0;
            for (int i = 0; i < a.n_pairs; ++i) {
                const int bb = a.pairs[2 * i], wi = a.pairs[2 * i + 1];
                if (bb != b) continue;
                if (wi < 0 || wi >= nw) {
                    set_status(C, QEVICT_ERR_STATE, a.layer, b, wi);
                    continue;
                }
                if (a.mode == PLAN_DEMOTE) {
                    // a listed demotion is to INT2; a window whose ledger has another width keeps it
                    if (s_cur[wi] != QEVICT_TIER_FP || (wi == nw - 1 && partial_last) ||
                        (D.lbits[wb + wi] != 0 && D.lbits[wb + wi] != 2)) {
                        set_status(C, QEVICT_ERR_STATE, a.layer, b, wi);
                        continue;
                    }
                    const int old_fp = D.fp_slot[wb + wi];
                    int lg = D.lg_slot[wb + wi];
                    if (lg < 0) {
                        const int top = ctr[CTR_LG_TOP];
                        if (top == 0) {
                            set_status(C, QEVICT_ERR_CAPACITY, a.layer, b, wi);
                            continue;
                        }
                        lg = D.lg_free[b * D.CQ + top - 1];
                        ctr[CTR_LG_TOP] = top - 1;
                        D.lg_slot[wb + wi] = lg;
                        D.lbits[wb + wi] = 2;
                        D.lwrites[wb + wi] += 1;
                        D.work_q[wb + nq++] = make_int4(wi, old_fp, lg, 2);
                        atomicAdd(&C.stats[ST_LWRITE], 1ull);
                    } else {
                        atomicAdd(&C.stats[ST_LREUSE], 1ull);
                    }
                    const int top = ctr[CTR_FP_TOP];
                    D.fp_free[b * D.CF + top] = old_fp;
                    ctr[CTR_FP_TOP] = top + 1;
                    D.fp_slot[wb + wi] = -1;
                    D.tier[wb + wi] = QEVICT_TIER_Q;
                    s_cur[wi] = QEVICT_TIER_Q;
                    atomicAdd(&C.stats[ST_DEMOTE], 1ull);
                } else {
                    if (!is_quant_tier(s_cur[wi])) {
                        set_status(C, QEVICT_ERR_STATE, a.layer, b, wi);
                        continue;
                    }
                    const int top = ctr[CTR_FP_TOP];
                    if (top == 0) {
                        set_status(C, QEVICT_ERR_CAPACITY, a.layer, b, wi);
                        continue;
                    }
                    const int fp = D.fp_free[b * D.CF + top - 1];
                    ctr[CTR_FP_TOP] = top - 1;
                    D.fp_slot[wb + wi] = fp;
                    D.tier[wb + wi] = QEVICT_TIER_FP;
                    D.work_p[wb + np++] = make_int4(wi, D.lg_slot[wb + wi], fp, D.lbits[wb + wi]);
                    s_cur[wi] = QEVICT_TIER_FP;
                    atomicAdd(&C.stats[ST_PROMOTE], 1ull);
                }
            }
            ctr[CTR_WQ] = nq;
            ctr[CTR_WP] = np;
        }
        __syncthreads();
        for (int i = tid; i < nw; i += kPlanThreads) s_tgt[i] = s_cur[i];
        __syncthreads();
    } else {
        // ---- target tiers
        for (int i = tid; i < nw; i += kPlanThreads) s_tgt[i] = s_cur[i];
        int bad = 0;
        if (a.mode == PLAN_ROUTE || a.mode == PLAN_PREFILL_SCORES || a.mode == PLAN_LOGSPARSE || a.mode == PLAN_RD ||
            a.mode == PLAN_RD_MIXED || a.mode == PLAN_RD_KV) {
            if (a.mode == PLAN_RD_KV) {
                // the K widths are set with the layer's first quantisation
                int has_ledger = 0;
                for (int i = tid; i < nw; i += kPlanThreads) has_ledger |= D.lg_slot[wb + i] >= 0;
                if (__syncthreads_or(has_ledger)) {
                    if (tid == 0) {
                        set_status(C, QEVICT_ERR_STATE, a.layer, b, -1);
                        reserve_next(D, ctr, b);
                    }
                    return;
                }
            }
            int P = 1;
            while (P < nw) P <<= 1;
            for (int i = tid; i < P; i += kPlanThreads) {
                unsigned long long key = ~0ull;
                if (i < nw && a.mode == PLAN_LOGSPARSE) {
                    // by position alone; the open window (age 0) ranks first; scores untouched
                    if (s_cur[i] != QEVICT_TIER_E)
                        key = ((unsigned long long)logsparse_rank(nw - 1 - i, a.recent) << 32) | (unsigned)i;
                } else if (i < nw) {
                    float S;
                    if (a.scores) {
                        S = a.scores[(int64_t)b * nw + i];
                    } else {
                        // the KV heads' partial scores, loaded together, added in head order
                        const float *spb = D.score_part + (int64_t)b * D.Hkv * D.Wmax + i;
                        float pv[8];
#pragma unroll
                        for (int h = 0; h < 8; ++h) pv[h] = h < D.Hkv ? spb[(int64_t)h * D.Wmax] : 0.f;
                        S = 0.f;
#pragma unroll
                        for (int h = 0; h < 8; ++h)
                            if (h < D.Hkv) S += pv[h];
                        for (int h = 8; h < D.Hkv; ++h) S += spb[(int64_t)h * D.Wmax];
                    }
                    if (a.mult) S = S * a.mult[(int64_t)b * nw + i];
                    if (S == 0.f) S = 0.f;   // one zero: -0 and +0 rank as equal
                    for (int h = 0; h < D.Hkv; ++h)
                        D.score_part[((int64_t)b * D.Hkv + h) * D.Wmax + i] = h == 0 ? S : 0.f;
                    if (s_cur[i] != QEVICT_TIER_E) {
                        if (!isfinite(S)) bad = 1;
                        key = (i == nw - 1) ? (unsigned long long)i
                                            : (((unsigned long long)(~orderable(S))) << 32) | (unsigned)i;
                    }
                }
                s_key[i] = key;
            }
            if (__syncthreads_or(bad)) {
                if (tid == 0) {
                    set_status(C, QEVICT_ERR_DEVICE, a.layer, b, -1);
                    reserve_next(D, ctr, b);
                }
                return;
            }
            // bitonic sort, ascending: forced window first, then score desc, index asc.
            // Strides of 32 and more exchange through shared memory; the smaller ones
            // pair lanes of one warp (index bits 0-4 are the lane) through shuffles.
            for (int kk = 2; kk <= P; kk <<= 1) {
                int j = kk >> 1;
                for (; j >= 32; j >>= 1) {
                    for (int i = tid; i < P; i += kPlanThreads) {
                        const int ixj = i ^ j;
                        if (ixj > i) {
                            const unsigned long long x = s_key[i], y = s_key[ixj];
                            const bool up = (i & kk) == 0;
                            if ((x > y) == up) {
                                s_key[i] = y;
                                s_key[ixj] = x;
                            }
                        }
                    }
                    __syncthreads();
                }
                for (int base = tid & ~31; base < P; base += kPlanThreads) {   // warp-uniform
                    const int i = base + (tid & 31);
                    unsigned long long x = i < P ? s_key[i] : ~0ull;
                    for (int jj = j; jj > 0; jj >>= 1) {
                        const unsigned ylo = __shfl_xor_sync(0xffffffffu, (unsigned)x, jj);
                        const unsigned yhi = __shfl_xor_sync(0xffffffffu, (unsigned)(x >> 32), jj);
                        const unsigned long long y = ((unsigned long long)yhi << 32) | ylo;
                        // the lower index of an ascending pair keeps the smaller key
                        const bool take_min = ((i & jj) == 0) == ((i & kk) == 0);
                        x = take_min ? (x < y ? x : y) : (x < y ? y : x);
                    }
                    if (i < P) s_key[i] = x;
                }
                __syncthreads();
            }
            int ncand_local = 0;
            for (int i = tid; i < nw; i += kPlanThreads) ncand_local += s_cur[i] != QEVICT_TIER_E;
            int ncand;
            block_scan(ncand_local, &ncand, s_warp);
            int n_fp, n_q;
            if (a.mode == PLAN_RD_MIXED || a.mode == PLAN_RD_KV) {
                rd_mixed_targets(D, s_key, s_tgt, ncand, budget, wb, s_warp, s_dyn);
                if (a.mode == PLAN_RD_KV) k_channel_widths(D, a.kweights, s_tgt, nw, b, s_warp);
                n_fp = n_q = -1;   // the targets are set
            } else if (a.mode == PLAN_RD) {
                // Rate-distortion counts. After the open window (rank 0) come upgrades
                // E -> INT2 of rank-i window (gain A[i] = alpha s_i, c_q bytes) and INT2 -> FP
                // (Q[i] = gamma s_i, c_fp - c_q bytes), taken in the merged order of the two
                // non-increasing lists (A first on a tie, then by rank) while positive, until the
                // first that does not fit. The taken ones are a prefix of the merged order, so each
                // upgrade finds its merged rank by binary search in the other list, adds up the cost
                // of the prefix through itself and decides alone. float64 gains, as the counts'
                // reference computes them.
                __shared__ double s_ag[2];   // the two gain factors, divided once by thread 0
                if (tid == 0) {
                    s_ag[0] = 0.75 / (double)D.c_q;
                    s_ag[1] = (0.25 - 1.52587890625e-05) / (double)(D.c_fp - D.c_q);
                }
                __syncthreads();
                const double alpha = s_ag[0], gamma = s_ag[1];
                auto score_at = [&](int i) { return key_score(s_key[1 + i]); };   // score of rank i + 1
                const int n = ncand - 1;
                const int64_t room = budget - D.c_fp;
                int up_local = 0, fp_local = 0;
                for (int e = tid; e < 2 * n; e += kPlanThreads) {
                    const bool is_q = e >= n;
                    const int i = is_q ? e - n : e;
                    const double v = (is_q ? gamma : alpha) * score_at(i);
                    if (!(v > 0.0)) continue;
                    // how many of the other list come before this one
                    int lo = 0, hi = n;
                    while (lo < hi) {
                        const int mid = (lo + hi) >> 1;
                        const double o = (is_q ? alpha : gamma) * score_at(mid);
                        if (is_q ? (o >= v) : (o > v))
                            lo = mid + 1;
                        else
                            hi = mid;
                    }
                    // prefix through this upgrade: EQ count and QF count
                    const int64_t n_eq = is_q ? lo : i + 1, n_qf = is_q ? i + 1 : lo;
                    if (n_eq * D.c_q + n_qf * (D.c_fp - D.c_q) <= room) {
                        if (is_q)
                            ++fp_local;
                        else
                            ++up_local;
                    }
                }
                int rd_v[2] = {up_local, fp_local}, rd_o[2], rd_t[2];
                block_scan_n<2>(rd_v, rd_o, rd_t, s_warp);
                const int up = rd_t[0], fp = rd_t[1];
                n_fp = ncand > 0 ? 1 + fp : 0;
                n_q = up - fp;
            } else {
                n_fp = min(ncand, max(1, nfp_budget));
                const int64_t rem = budget - (int64_t)n_fp * D.c_fp;
                n_q = (int)min((int64_t)(ncand - n_fp), rem > 0 ? rem / D.c_q : 0);
            }
            for (int r = tid; r < ncand && n_fp >= 0; r += kPlanThreads) {
                const int wi = (int)(s_key[r] & 0xffffffffu);
                s_tgt[wi] = r < n_fp ? QEVICT_TIER_FP : (r < n_fp + n_q ? QEVICT_TIER_Q : QEVICT_TIER_E);
            }
            __syncthreads();
        } else if (a.mode == PLAN_GLOBAL) {
            // the sequence's keys across all layers were ranked by global_select_kernel:
            // classify this layer's candidates against its two thresholds
            const int seq = b / D.hs, j = b % D.hs;
            if (a.gflag[seq] == 0) {   // the event stopped on an error, reported by the select kernel
                if (tid == 0) reserve_next(D, ctr, b);
                return;
            }
            const unsigned long long t_fp = a.gthr[2 * seq], t_q = a.gthr[2 * seq + 1];
            const unsigned long long *keys =
                a.gkeys + ((int64_t)seq * a.glayers * D.hs + (int64_t)a.layer * D.hs + j) * D.Wmax;
            for (int i = tid; i < nw; i += kPlanThreads) {
                if (s_cur[i] == QEVICT_TIER_E) continue;
                const unsigned long long k = keys[i];
                s_tgt[i] = k >= t_fp ? QEVICT_TIER_FP : (k >= t_q ? QEVICT_TIER_Q : QEVICT_TIER_E);
            }
            __syncthreads();
        } else {
            for (int i = tid; i < nw; i += kPlanThreads) {
                const uint8_t t = a.tiers[(int64_t)b * nw + i];
                const uint8_t c = s_cur[i];
                const int lb = prefill ? 0 : D.lbits[wb + i];
                const bool allowed = t <= QEVICT_TIER_E || (t == QEVICT_TIER_Q4 && D.maxP >= 2) ||
                                     (t == QEVICT_TIER_Q8 && D.maxP >= 4);
                if (!allowed || (c == QEVICT_TIER_E && t != QEVICT_TIER_E) ||
                    (i == nw - 1 && partial_last && t != c) ||
                    (is_quant_tier(c) && is_quant_tier(t) && c != t) ||   // a quantised window keeps its width
                    (c == QEVICT_TIER_FP && is_quant_tier(t) && lb != 0 && lb != tier_bits(t)))   // so does its ledger
                    bad = 1;
                s_tgt[i] = t;
            }
            if (__syncthreads_or(bad)) {
                if (tid == 0) {
                    set_status(C, QEVICT_ERR_STATE, a.layer, b, -1);
                    reserve_next(D, ctr, b);
                }
                return;
            }
        }

        // ---- capacity check
        const int per = (nw + kPlanThreads - 1) / kPlanThreads;
        const int w0 = tid * per, w1 = min(nw, w0 + per);
        int free_fp = 0, free_lg = 0, need_fp = 0, need_lg = 0;
        for (int i = w0; i < w1; ++i) {
            const uint8_t c = s_cur[i], t = s_tgt[i];
            const int lg = prefill ? -1 : D.lg_slot[wb + i];
            if (!prefill && c == QEVICT_TIER_FP && t != QEVICT_TIER_FP) ++free_fp;
            if (c != QEVICT_TIER_E && t == QEVICT_TIER_E && lg >= 0) ++free_lg;
            if (c == QEVICT_TIER_FP && is_quant_tier(t) && lg < 0) ++need_lg;
            if ((is_quant_tier(c) && t == QEVICT_TIER_FP) || (prefill && t == QEVICT_TIER_FP)) ++need_fp;
        }
        int cap_v[4] = {free_fp, free_lg, need_fp, need_lg}, cap_o[4], cap_t[4];
        block_scan_n<4>(cap_v, cap_o, cap_t, s_warp);
        const int off_free_fp = cap_o[0], off_free_lg = cap_o[1], off_need_fp = cap_o[2], off_need_lg = cap_o[3];
        const int tot_free_fp = cap_t[0], tot_free_lg = cap_t[1], tot_need_fp = cap_t[2], tot_need_lg = cap_t[3];
        const int fp_top = ctr[CTR_FP_TOP], lg_top = ctr[CTR_LG_TOP];
        if (fp_top + tot_free_fp < tot_need_fp || lg_top + tot_free_lg < tot_need_lg) {
            if (tid == 0) {
                set_status(C, QEVICT_ERR_CAPACITY, a.layer, b, -1);
                reserve_next(D, ctr, b);
            }
            return;
        }
        // ---- phase A: release slots
        {
            int of = off_free_fp, ol = off_free_lg;
            for (int i = w0; i < w1; ++i) {
                const uint8_t c = s_cur[i], t = s_tgt[i];
                if (!prefill && c == QEVICT_TIER_FP && t != QEVICT_TIER_FP)
                    D.fp_free[b * D.CF + fp_top + of++] = D.fp_slot[wb + i];
                const int lg = prefill ? -1 : D.lg_slot[wb + i];
                if (c != QEVICT_TIER_E && t == QEVICT_TIER_E && lg >= 0)
                    D.lg_free[b * D.CQ + lg_top + ol++] = lg;
            }
        }
        __syncthreads();
        const int fp_mid = fp_top + tot_free_fp, lg_mid = lg_top + tot_free_lg;
        // ---- phase B: take slots, update the table, queue data movement
        int nq_local = 0, np_local = 0, nc_local = 0;
        for (int i = w0; i < w1; ++i) {
            const uint8_t c = s_cur[i], t = s_tgt[i];
            nq_local += (c == QEVICT_TIER_FP && is_quant_tier(t) && (prefill || D.lg_slot[wb + i] < 0));
            np_local += (!prefill && is_quant_tier(c) && t == QEVICT_TIER_FP);
            nc_local += (prefill && t == QEVICT_TIER_FP);
        }
        int mv_v[3] = {nq_local, np_local, nc_local}, mv_o[3], mv_t[3];
        block_scan_n<3>(mv_v, mv_o, mv_t, s_warp);
        int oq = mv_o[0], op = mv_o[1], oc = mv_o[2];
        const int tq = mv_t[0], tp = mv_t[1], tc = mv_t[2];
        int nf = off_need_fp, nl = off_need_lg;
        unsigned long long st_dem = 0, st_pro = 0, st_evi = 0, st_lw = 0, st_lr = 0;
        for (int i = w0; i < w1; ++i) {
            const uint8_t c = s_cur[i], t = s_tgt[i];
            const int64_t e = wb + i;
            if (prefill) {
                D.lwrites[e] = 0;
                D.lg_slot[e] = -1;
                D.fp_slot[e] = -1;
                D.lbits[e] = 0;
                if (t == QEVICT_TIER_FP) {
                    const int fp = D.fp_free[b * D.CF + fp_mid - 1 - nf++];
                    D.fp_slot[e] = fp;
                    D.work_c[wb + oc++] = make_int4(i, fp, 0, 0);
                } else if (is_quant_tier(t)) {
                    const int lg = D.lg_free[b * D.CQ + lg_mid - 1 - nl++];
                    D.lg_slot[e] = lg;
                    D.lbits[e] = (uint8_t)tier_bits(t);
                    D.lwrites[e] = 1;
                    D.work_q[wb + oq++] = make_int4(i, -1, lg, tier_bits(t));
                    ++st_dem;
                    ++st_lw;
                } else {
                    ++st_evi;
                }
                D.tier[e] = t;
                for (int h = 0; h < D.Hkv; ++h)
                    if (a.mode == PLAN_PREFILL_TIERS) D.score_part[((int64_t)b * D.Hkv + h) * D.Wmax + i] = 0.f;
                continue;
            }
            if (c == t) continue;
            if (t == QEVICT_TIER_E) {
                D.fp_slot[e] = -1;
                D.lg_slot[e] = -1;
                D.lbits[e] = 0;
                ++st_evi;
            } else if (c == QEVICT_TIER_FP && is_quant_tier(t)) {
                const int old_fp = D.fp_slot[e];
                if (D.lg_slot[e] < 0) {
                    const int lg = D.lg_free[b * D.CQ + lg_mid - 1 - nl++];
                    D.lg_slot[e] = lg;
                    D.lbits[e] = (uint8_t)tier_bits(t);
                    D.lwrites[e] += 1;
                    D.work_q[wb + oq++] = make_int4(i, old_fp, lg, tier_bits(t));
                    ++st_lw;
                } else {
                    ++st_lr;
                }
                D.fp_slot[e] = -1;
                ++st_dem;
            } else if (is_quant_tier(c) && t == QEVICT_TIER_FP) {
                const int fp = D.fp_free[b * D.CF + fp_mid - 1 - nf++];
                D.fp_slot[e] = fp;
                D.work_p[wb + op++] = make_int4(i, D.lg_slot[e], fp, D.lbits[e]);
                ++st_pro;
            }
            D.tier[e] = t;
        }
        if (st_dem) atomicAdd(&C.stats[ST_DEMOTE], st_dem);
        if (st_pro) atomicAdd(&C.stats[ST_PROMOTE], st_pro);
        if (st_evi) atomicAdd(&C.stats[ST_EVICT], st_evi);
        if (st_lw) atomicAdd(&C.stats[ST_LWRITE], st_lw);
        if (st_lr) atomicAdd(&C.stats[ST_LREUSE], st_lr);
        if (tid == 0) {
            ctr[CTR_FP_TOP] = fp_mid - tot_need_fp;
            ctr[CTR_LG_TOP] = lg_mid - tot_need_lg;
            ctr[CTR_WQ] = tq;
            ctr[CTR_WP] = tp;
            ctr[CTR_WC] = tc;
        }
        __syncthreads();
    }

    // ---- rebuild the per-tier window lists
    const int per = (nw + kPlanThreads - 1) / kPlanThreads;
    const int w0 = tid * per, w1 = min(nw, w0 + per);
    int nfp_local = 0, nq_local = 0;
    for (int i = w0; i < w1; ++i) {
        nfp_local += s_tgt[i] == QEVICT_TIER_FP;
        nq_local += is_quant_tier(s_tgt[i]);
    }
    int ls_v[2] = {nfp_local, nq_local}, ls_o[2], ls_t[2];
    block_scan_n<2>(ls_v, ls_o, ls_t, s_warp);
    int of = ls_o[0], oq = ls_o[1];
    const int tf = ls_t[0], tq = ls_t[1];
    for (int i = w0; i < w1; ++i) {
        if (s_tgt[i] == QEVICT_TIER_FP) D.fp_list[b * D.CF + of++] = make_int2(i, D.fp_slot[wb + i]);
        if (is_quant_tier(s_tgt[i])) {   // the slot field carries log2 of the window's planes
            const int lb = D.lbits[wb + i];
            D.q_list[b * D.CQ + oq++] = make_int2(i, D.lg_slot[wb + i] | ((lb == 8 ? 2 : lb == 4 ? 1 : 0) << kSlotBits));
        }
    }
    // ---- the move's counts (the full-precision tier read as the active set):
    // tier sizes before and after, kept, promoted, demoted, evicted
    {
        int cnt[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int i = w0; i < w1; ++i) {
            const uint8_t o = s_old[i], n = s_tgt[i];
            cnt[0] += o == QEVICT_TIER_FP;
            cnt[1] += is_quant_tier(o);
            cnt[2] += n == QEVICT_TIER_FP;
            cnt[3] += is_quant_tier(n);
            cnt[4] += o == QEVICT_TIER_FP && n == QEVICT_TIER_FP;
            cnt[5] += is_quant_tier(o) && n == QEVICT_TIER_FP;
            cnt[6] += o == QEVICT_TIER_FP && is_quant_tier(n);
            cnt[7] += o != QEVICT_TIER_E && n == QEVICT_TIER_E;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (cnt[j]) atomicAdd(&s_cnt[j], cnt[j]);
        __syncthreads();
        if (tid < 8) D.diag[b * 8 + tid] = s_cnt[tid];
    }
    if (tid == 0) {
        ctr[CTR_NFP] = tf;
        ctr[CTR_NQ] = tq;
        if (prefill) ctr[CTR_LEN] = (int)length;
        reserve_next(D, ctr, b);
    }
}

// ---------------------------------------------------------------- quantise
// INT2 quantisation of one window part (entry, KV head, K or V): per token and
// group of 32 channels, min16 = fp16(min), scale16 = fp16(fl32(fl32(max-min)/3)),
// code = clamp(rint(fl32(fl32(x - min16) / scale16)), 0, 3). The rounded
// quotient comes from the scale's rounded reciprocal and an FMA correction
// (div_by_recip), not from a division per element.
__global__ void __launch_bounds__(128) quantize_kernel(LayerDev D, CacheDev C, int layer,
                                                        const __nv_bfloat16 *__restrict__ k_ext,
                                                        const __nv_bfloat16 *__restrict__ v_ext,
                                                        int64_t ext_len) {
    extern __shared__ uint8_t s_codes[];   // [w][d]
    const int b = blockIdx.z;
    const int h = blockIdx.y >> 1, kv = blockIdx.y & 1;
    const int w = D.w;
    const int n = D.ctr[b * kCtrN + CTR_WQ];
    // a K-channel layer: K group widths of this KV head, and the tiles' K code bytes
    const bool kch = D.ctr[b * kCtrN + CTR_KCH] != 0;
    const uint8_t *kw = kch ? D.kgw + ((int64_t)b * D.Hkv + h) * kGroups : nullptr;
    const int kcodes = kch ? ktile_kcodes(kw) : 0;
    for (int e = blockIdx.x; e < n; e += gridDim.x) {
        const int4 job = D.work_q[(int64_t)b * D.Wmax + e];
        const int wi = job.x, src_slot = job.y, dst = job.z;
        // the width: 2, 4 or 8 bits, written as P 2-bit planes
        const int bits = job.w == 4 || job.w == 8 ? job.w : 2, P = bits / 2;
        uint8_t *slotp = D.lg_pool + (int64_t)dst * D.lg_slot_bytes;
        // tile offsets in the slot, and the meta of this part within a tile
        const int tstride = kch ? qtile_bytes(4) : qtile_bytes(P);
        const int meta_off = kch ? (kv ? kcodes + 256 + 512 * P : kcodes) : (kv ? qtile_vmeta(P) : qtile_kmeta(P));
        for (int it = threadIdx.x; it < w * kGroups; it += blockDim.x) {
            const int t = it / kGroups, g = it % kGroups;
            // K groups of a K-channel layer take their own widths; width 0 keeps no codes
            const int gbits = (kw && kv == 0) ? kw[g] : bits;
            const float levels = (float)((1 << (gbits > 0 ? gbits : 2)) - 1);
            const __nv_bfloat16 *src;
            if (src_slot >= 0) {
                src = reinterpret_cast<const __nv_bfloat16 *>(D.fp_pool + (int64_t)src_slot * D.fp_slot_bytes) +
                      fp_off(h, kv, w, t, g * kGroup);
            } else {
                src = (kv ? v_ext : k_ext) + src_row(D, b, ext_len, (int64_t)wi * w + t, h) * kHeadDim + g * kGroup;
            }
            // the group's minimum and maximum on bf16 pairs, with NaN propagating, so that
            // a NaN or an infinity anywhere in the group shows in them
            float x[kGroup];
            __nv_bfloat162 mn2, mx2;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 u = reinterpret_cast<const uint4 *>(src)[c];
                const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 f = __bfloat1622float2(p2[j]);
                    x[c * 8 + 2 * j] = f.x;
                    x[c * 8 + 2 * j + 1] = f.y;
                    mn2 = (c == 0 && j == 0) ? p2[j] : __hmin2_nan(mn2, p2[j]);
                    mx2 = (c == 0 && j == 0) ? p2[j] : __hmax2_nan(mx2, p2[j]);
                }
            }
            const float mn = __bfloat162float(__hmin_nan(__low2bfloat16(mn2), __high2bfloat16(mn2)));
            const float mx = __bfloat162float(__hmax_nan(__low2bfloat16(mx2), __high2bfloat16(mx2)));
            const bool finite = isfinite(mn) && isfinite(mx);
            const __half mn16 = __float2half_rn(mn);
            const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), levels));
            const float mq = __half2float(mn16), sq = __half2float(s16);
            const bool bad = gbits > 0 && (!finite || isinf(mq) || isinf(sq));
            if (bad) set_status(C, QEVICT_ERR_DEVICE, layer, b, wi);
            const bool zero = bad || sq == 0.f || gbits == 0;
            // the quotients through the scale's reciprocal, corrected to the rounded quotient;
            // clamped to [0, levels] (0 for a zero scale), then rounded half to even by adding
            // 1.5 * 2^23, whose float has the integer in its low mantissa bits (clamping first
            // gives the same code as rounding first)
            const float sdiv = zero ? 1.f : sq;
            const float rs = __frcp_rn(sdiv);
            const float top = zero ? 0.f : levels;
            uint32_t *cs = reinterpret_cast<uint32_t *>(s_codes + t * kHeadDim + g * kGroup);
#pragma unroll
            for (int j = 0; j < kGroup; j += 4) {
                uint32_t c4[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float qv = fminf(fmaxf(div_by_recip(__fsub_rn(x[j + k], mq), sdiv, rs), 0.f), top);
                    c4[k] = __float_as_uint(__fadd_rn(qv, 12582912.f));
                }
                cs[j / 4] = __byte_perm(__byte_perm(c4[0], c4[1], 0x0040), __byte_perm(c4[2], c4[3], 0x0040), 0x5410);
            }
            __half2 *meta = reinterpret_cast<__half2 *>(slotp + ((int64_t)h * (w / 16) + t / 16) * tstride + meta_off) +
                            (t % 16) * kGroups + g;
            *meta = (bad || gbits == 0) ? __halves2half2(__float2half_rn(0.f), __float2half_rn(0.f))
                                        : __halves2half2(s16, mn16);
        }
        __syncthreads();
        if (kv == 0 && kw) {
            // K of a K-channel layer: group g's planes in turn, each [16 tokens][2 words of 16
            // channels], channel j of a word at bits 2*(j%16), plane p holding bits 2p, 2p + 1
            int goff = 0;
            for (int g = 0; g < kGroups; ++g) {
                const int Pg = kgroup_planes(kw[g]);
                for (int i = threadIdx.x; i < Pg * w * 2; i += blockDim.x) {
                    const int p = i / (w * 2), r = i % (w * 2), t = r / 2, hq = r % 2;
                    const uint8_t *cs = s_codes + t * kHeadDim + g * kGroup + hq * 16;
                    uint32_t word = 0;
#pragma unroll
                    for (int j = 0; j < 16; ++j) word |= (uint32_t)((cs[j] >> (2 * p)) & 3u) << (2 * j);
                    reinterpret_cast<uint32_t *>(slotp + ((int64_t)h * (w / 16) + t / 16) * tstride + goff + 128 * p)
                        [(t % 16) * 2 + hq] = word;
                }
                goff += 128 * Pg;
            }
        } else if (kv == 0) {
            // K: per token 8 words of 16 channels, channel j of the word at bits 2*(j%16); plane p
            // of a wider code holds its bits 2p, 2p + 1
            for (int i = threadIdx.x; i < P * w * (kHeadDim / 16); i += blockDim.x) {
                const int p = i / (w * (kHeadDim / 16)), r = i % (w * (kHeadDim / 16));
                const int t = r / (kHeadDim / 16), q = r % (kHeadDim / 16);
                const uint8_t *cs = s_codes + t * kHeadDim + q * 16;
                uint32_t word = 0;
#pragma unroll
                for (int j = 0; j < 16; ++j) word |= (uint32_t)((cs[j] >> (2 * p)) & 3u) << (2 * j);
                reinterpret_cast<uint32_t *>(slotp + lg_tile_off(h, w, t / 16, P) + 512 * p)[(t % 16) * 8 + q] = word;
            }
        } else {
            // V: per 16-token tile 128 words; word i holds channel vword_dim(i), token t of
            // the tile at bits 2*(t%16); plane p of a wider code holds its bits 2p, 2p + 1
            for (int i = threadIdx.x; i < P * (w / kVTile) * kHeadDim; i += blockDim.x) {
                const int p = i / ((w / kVTile) * kHeadDim), r = i % ((w / kVTile) * kHeadDim);
                const int tile = r / kHeadDim, j = vword_dim(r % kHeadDim);
                uint32_t word = 0;
#pragma unroll
                for (int t = 0; t < kVTile; ++t)
                    word |= (uint32_t)((s_codes[(tile * kVTile + t) * kHeadDim + j] >> (2 * p)) & 3u) << (2 * t);
                const int vcodes = kw ? kcodes + 256 : qtile_vcodes(P);
                reinterpret_cast<uint32_t *>(slotp + ((int64_t)h * (w / 16) + tile) * tstride + vcodes + 512 * p)
                    [r % kHeadDim] = word;
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- promote
// bf16_rne(fmaf(code, scale, min)) from a ledger part into a full-precision slot.
__global__ void __launch_bounds__(128) promote_kernel(LayerDev D) {
    const int b = blockIdx.z;
    const int h = blockIdx.y >> 1, kv = blockIdx.y & 1;
    const int w = D.w;
    const int n = D.ctr[b * kCtrN + CTR_WP];
    // one 16-token tile of this (KV head, K or V) at a time: its code words
    // (128 per plane) and 64 (scale, min) pairs staged with coalesced loads
    __shared__ uint32_t s_codes[4][128];
    __shared__ __half2 s_meta[64];
    const int tid = threadIdx.x;
    for (int e = blockIdx.x; e < n; e += gridDim.x) {
        const int4 job = D.work_p[(int64_t)b * D.Wmax + e];
        const int P = job.w == 4 ? 2 : (job.w == 8 ? 4 : 1);   // planes of the window's ledger width
        const uint8_t *slotp = D.lg_pool + (int64_t)job.y * D.lg_slot_bytes;
        __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(D.fp_pool + (int64_t)job.z * D.fp_slot_bytes);
        for (int tile = 0; tile < w / 16; ++tile) {
            const uint8_t *tp = slotp + lg_tile_off(h, w, tile, P);
            __syncthreads();   // the previous tile's values are used up
            for (int p = 0; p < P; ++p)
                s_codes[p][tid] = reinterpret_cast<const uint32_t *>(tp + (kv ? qtile_vcodes(P) : 0) + 512 * p)[tid];
            if (tid < 64)
                s_meta[tid] = reinterpret_cast<const __half2 *>(tp + (kv ? qtile_vmeta(P) : qtile_kmeta(P)))[tid];
            __syncthreads();
            // 16 tokens x 16 runs of 8 channels: two (token, run) items per thread
            for (int it = tid; it < 16 * 16; it += 128) {
                const int t = it >> 4, ch0 = (it & 15) * 8;
                const __half2 m2 = s_meta[t * kGroups + ch0 / kGroup];
                const float sc = __low2float(m2), mn = __high2float(m2);
                __align__(16) __nv_bfloat16 outv[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int ch = ch0 + j;
                    uint32_t c = 0;
                    for (int p = 0; p < P; ++p)   // code = sum_p 4^p c_p
                        c |= (kv == 0 ? (s_codes[p][t * 8 + ch / 16] >> (2 * (ch % 16))) & 3u
                                      : (s_codes[p][vword_index(ch)] >> (2 * (t % kVTile))) & 3u)
                             << (2 * p);
                    outv[j] = __float2bfloat16_rn(fmaf((float)c, sc, mn));
                }
                *reinterpret_cast<uint4 *>(dst + fp_off(h, kv, w, tile * 16 + t, ch0)) =
                    *reinterpret_cast<const uint4 *>(outv);
            }
        }
    }
}

// ---------------------------------------------------------------- prefill copy
__global__ void __launch_bounds__(128) prefill_copy_kernel(LayerDev D, const __nv_bfloat16 *__restrict__ k_ext,
                                                            const __nv_bfloat16 *__restrict__ v_ext,
                                                            int64_t ext_len) {
    const int b = blockIdx.z;
    const int h = blockIdx.y >> 1, kv = blockIdx.y & 1;
    const int w = D.w;
    const int n = D.ctr[b * kCtrN + CTR_WC];
    constexpr int kChunks = kHeadDim * 2 / 16;
    for (int e = blockIdx.x; e < n; e += gridDim.x) {
        const int4 job = D.work_c[(int64_t)b * D.Wmax + e];
        const int wi = job.x;
        const int ntok = (int)min((int64_t)w, ext_len - (int64_t)wi * w);
        __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(D.fp_pool + (int64_t)job.y * D.fp_slot_bytes);
        const __nv_bfloat16 *srcb = kv ? v_ext : k_ext;
        for (int i = threadIdx.x; i < ntok * kChunks; i += blockDim.x) {
            const int t = i / kChunks, c = i % kChunks;
            const __nv_bfloat16 *src = srcb + src_row(D, b, ext_len, (int64_t)wi * w + t, h) * kHeadDim;
            *reinterpret_cast<uint4 *>(dst + fp_off(h, kv, w, t, 8 * c)) = reinterpret_cast<const uint4 *>(src)[c];
        }
    }
}

// Every sequence of the batch has the same length; report sequence 0's.
__global__ void read_lengths_kernel(LayerDev D, int32_t *out) {
    if (threadIdx.x == 0) out[0] = D.ctr[CTR_LEN];
}

__global__ void scores_kernel(LayerDev D, int n_win, float *out) {
    const int64_t n = (int64_t)D.B * n_win;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int b = (int)(i / n_win), wi = (int)(i % n_win);
        float s = 0.f;
        for (int h = 0; h < D.Hkv; ++h) s += D.score_part[((int64_t)b * D.Hkv + h) * D.Wmax + wi];
        out[i] = s;
    }
}

// ---------------------------------------------------------------- global routing
// Ranking key of a candidate window of a global routing event: larger ranks
// first. Forced (the last window of each unit of each layer) above everything,
// then the score, then the lower (layer, unit, window) index. Unique within a
// sequence, and never 0 (0 marks a non-candidate).
__device__ __forceinline__ unsigned long long global_key(float S, bool forced, uint32_t gidx) {
    return ((unsigned long long)(forced ? 0xffffffffu : orderable(S)) << 32) | (0xffffffffu - gidx);
}

// Of the 256 digit bins (counts h[d]), the digit of the K-th largest key among
// those in the bins, with *rem = K on entry and K's rank inside that bin on
// exit. Warp-wide: lane L sums bins 255 - 8L down to 248 - 8L.
__device__ __forceinline__ int top_bin(const unsigned *h, long long *rem, int lane) {
    unsigned part = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) part += h[255 - 8 * lane - i];
    unsigned incl = part;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const long long r = *rem;
    const unsigned ball = __ballot_sync(0xffffffffu, (long long)incl >= r);
    const int L = __ffs(ball) - 1;   // the first lane whose bins reach rank r
    int digit = 0;
    long long left = 0;
    if (lane == L) {
        long long cum = (long long)(incl - part);
        for (int i = 0; i < 8; ++i) {
            const int d = 255 - 8 * lane - i;
            if (cum + h[d] >= r) {
                digit = d;
                left = r - cum;
                break;
            }
            cum += h[d];
        }
    }
    digit = __shfl_sync(0xffffffffu, digit, L);
    left = __shfl_sync(0xffffffffu, left, L);
    *rem = left;
    return digit;
}

// Keys of a global routing event: one CTA per (range of 1024 entries of a
// layer's [hs][Wmax] table, layer, sequence). Writes the ranking key of every
// candidate window (0 elsewhere), collapsing each score's per-KV-head
// partials into one value as a per-layer route does, and adds the sequence's
// candidate, forced and non-finite counts to g.cnt.
__global__ void __launch_bounds__(1024) global_keys_kernel(GlobalArgs g) {
    const int l = blockIdx.y, seq = blockIdx.z, tid = threadIdx.x;
    const int64_t per_layer = (int64_t)g.hs * g.Wmax;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + tid;
    const LayerDev &D = g.layers[l];
    const int u0 = seq * g.hs;
    const int64_t len = D.ctr[u0 * kCtrN + CTR_LEN];
    const int nw = (int)((len + g.w - 1) / g.w);
    int cand = 0, forced = 0, bad = 0;
    if (i < per_layer) {
        const int j = (int)(i / g.Wmax), wi = (int)(i % g.Wmax), u = u0 + j;
        unsigned long long key = 0;
        if (wi < nw && D.tier[(int64_t)u * D.Wmax + wi] != QEVICT_TIER_E) {
            float S = 0.f;
            for (int h = 0; h < D.Hkv; ++h) S += D.score_part[((int64_t)u * D.Hkv + h) * D.Wmax + wi];
            if (S == 0.f) S = 0.f;   // one zero: -0 and +0 rank as equal
            for (int h = 0; h < D.Hkv; ++h) D.score_part[((int64_t)u * D.Hkv + h) * D.Wmax + wi] = h == 0 ? S : 0.f;
            bad = !isfinite(S);
            const bool f = wi == nw - 1;
            key = global_key(S, f, (uint32_t)(l * per_layer + i));
            cand = 1;
            forced = f;
        }
        g.keys[((int64_t)seq * g.num_layers + l) * per_layer + i] = key;
    }
    cand = __reduce_add_sync(0xffffffffu, cand);
    forced = __reduce_add_sync(0xffffffffu, forced);
    bad = __reduce_or_sync(0xffffffffu, bad);
    if ((tid & 31) == 0 && (cand | bad)) {
        atomicAdd(&g.cnt[4 * seq], cand);
        atomicAdd(&g.cnt[4 * seq + 1], forced);
        if (bad) atomicOr(&g.cnt[4 * seq + 2], 1);
    }
}

// One cluster of kSelCtas CTAs per sequence, after global_keys_kernel: the
// one budget and the counts, then the n_fp-th and (n_fp + n_q)-th largest
// keys by radix selection (8 passes of 8 bits). Each CTA histograms its
// eighth of the sequence's key table in its own shared memory and adds it
// into rank 0's through distributed shared memory; rank 0 picks each pass's
// digits. Leaves the sequence's counters at zero for the next event.
constexpr int kSelCtas = 8;

__global__ void __cluster_dims__(kSelCtas, 1, 1) __launch_bounds__(1024)
    global_select_kernel(GlobalArgs g, CacheDev C) {
    cg::cluster_group cl = cg::this_cluster();
    const int rank = (int)cl.block_rank();
    const int seq = blockIdx.x / kSelCtas, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __shared__ unsigned s_h[2][256];    // this CTA's histograms
    __shared__ unsigned s_hc[2][256];   // rank 0: the cluster's
    __shared__ int s_go;
    __shared__ unsigned long long s_pre[2];
    __shared__ long long s_rem[2];
    const int64_t per_seq = (int64_t)g.num_layers * g.hs * g.Wmax;
    const unsigned long long *keys = g.keys + (int64_t)seq * per_seq;
    if (rank == 0 && tid == 0) {
        int go = 1;
        int64_t F = 0;
        for (int l = 0; l < g.num_layers; ++l) {
            const LayerDev &D = g.layers[l];
            F += (int64_t)g.hs * D.ctr[seq * g.hs * kCtrN + CTR_LEN] * D.Hkv * kHeadDim * 4;
        }
        const int64_t Bg = (int64_t)floor(g.beta * (double)F);
        const int C_ = g.cnt[4 * seq], nf = g.cnt[4 * seq + 1], bad = g.cnt[4 * seq + 2];
        g.cnt[4 * seq] = 0;
        g.cnt[4 * seq + 1] = 0;
        g.cnt[4 * seq + 2] = 0;
        int n_fp = 0, n_q = 0;
        if (bad) {
            set_status(C, QEVICT_ERR_DEVICE, -1, seq, -1);
            go = 0;
        } else if ((int64_t)nf * g.c_fp > Bg) {
            set_status(C, QEVICT_ERR_BUDGET, -1, seq, nf);
            go = 0;
        } else {
            const int nfp_budget = (int)floor((g.rho * (double)Bg) / (double)g.c_fp);
            n_fp = min(C_, max(nf, nfp_budget));
            const int64_t rem = Bg - (int64_t)n_fp * g.c_fp;
            n_q = (int)min((int64_t)(C_ - n_fp), rem > 0 ? rem / g.c_q : 0);
        }
        g.flag[seq] = go;
        s_rem[0] = n_fp;
        s_rem[1] = (long long)n_fp + n_q;
        s_pre[0] = 0;
        s_pre[1] = 0;
        s_go = go;
    }
    cl.sync();
    int *go0 = cl.map_shared_rank(&s_go, 0);
    long long *rem0 = cl.map_shared_rank(&s_rem[0], 0);
    unsigned long long *pre0 = cl.map_shared_rank(&s_pre[0], 0);
    unsigned *hc0 = cl.map_shared_rank(&s_hc[0][0], 0);
    const bool go = *go0 != 0;
    // rank 0 zero (no candidates) selects nothing
    const bool want0 = rem0[0] > 0, want1 = rem0[1] > 0;
    cl.sync();   // every CTA has read rank 0's start values
    if (!go) return;
    const int64_t i_lo = per_seq * rank / kSelCtas, i_hi = per_seq * (rank + 1) / kSelCtas;
    unsigned long long mask = 0;
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = tid; i < 512; i += blockDim.x) {
            (&s_h[0][0])[i] = 0;
            if (rank == 0) (&s_hc[0][0])[i] = 0;
        }
        const unsigned long long p0 = pre0[0], p1 = pre0[1];
        cl.sync();   // rank 0's bins are zero before anyone adds
        for (int64_t i0 = i_lo + tid; i0 < i_hi; i0 += 8 * (int64_t)blockDim.x) {
            unsigned long long kk[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t i = i0 + (int64_t)u * blockDim.x;
                kk[u] = i < i_hi ? __ldcg(keys + i) : 0ull;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const unsigned long long k = kk[u];
                if (!k) continue;
                const unsigned d = (unsigned)(k >> shift) & 255u;
                if ((k & mask) == p0) atomicAdd(&s_h[0][d], 1u);
                if ((k & mask) == p1) atomicAdd(&s_h[1][d], 1u);
            }
        }
        __syncthreads();
        for (int i = tid; i < 512; i += blockDim.x) {
            const unsigned v = (&s_h[0][0])[i];
            if (v) atomicAdd(hc0 + i, v);
        }
        cl.sync();   // the cluster's histograms are complete
        if (rank == 0 && warp < 2 && (warp == 0 ? want0 : want1)) {
            long long r = s_rem[warp];
            const int d = top_bin(s_hc[warp], &r, lane);
            if (lane == 0) {
                s_rem[warp] = r;
                s_pre[warp] |= (unsigned long long)d << shift;
            }
        }
        mask |= 0xffull << shift;
        cl.sync();   // the digits are in rank 0's shared memory
    }
    if (rank == 0 && tid == 0) {
        // no rank asked: a threshold above every key
        g.thr[2 * seq] = want0 ? s_pre[0] : ~0ull;
        g.thr[2 * seq + 1] = want1 ? s_pre[1] : ~0ull;
    }
}

__global__ void set_scores_kernel(LayerDev D, const float *scores, int n_win) {
    const int64_t n = (int64_t)D.B * n_win;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int u = (int)(i / n_win), wi = (int)(i % n_win);
        for (int h = 0; h < D.Hkv; ++h)
            D.score_part[((int64_t)u * D.Hkv + h) * D.Wmax + wi] = h == 0 ? scores[i] : 0.f;
    }
}

}  // namespace

cudaError_t launch_global_select(const GlobalArgs &g, const CacheDev &C, int sequences, cudaStream_t s) {
    const int64_t per_layer = (int64_t)g.hs * g.Wmax;
    global_keys_kernel<<<dim3((unsigned)((per_layer + 1023) / 1024), g.num_layers, sequences), 1024, 0, s>>>(g);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    global_select_kernel<<<sequences * kSelCtas, 1024, 0, s>>>(g, C);
    return cudaGetLastError();
}

cudaError_t launch_set_scores(const LayerDev &L, const float *scores, int n_win, cudaStream_t s) {
    set_scores_kernel<<<64, 256, 0, s>>>(L, scores, n_win);
    return cudaGetLastError();
}

cudaError_t launch_init_layer(const LayerDev &L, cudaStream_t s) {
    init_layer_kernel<<<256, 256, 0, s>>>(L);
    return cudaGetLastError();
}

cudaError_t launch_append(const LayerDev &L, const CacheDev &C, int layer, const __nv_bfloat16 *k,
                          const __nv_bfloat16 *v, int n_new, cudaStream_t s) {
    append_kernel<<<L.B, 256, 0, s>>>(L, C, layer, k, v, n_new);
    return cudaGetLastError();
}

// Dynamic shared memory of the mixed-width route: one 8-byte gain per chain step
// of every window (a never-quantised window has the most steps), then one
// 2-byte rank index per window.
static size_t mixed_plan_smem(const LayerDev &L) {
    const int steps = 2 + (L.maxP >= 2) + (L.maxP >= 4);
    return (size_t)steps * L.Wmax * 8 + (size_t)L.Wmax * 2;
}

cudaError_t launch_plan(const LayerDev &L, const CacheDev &C, const PlanArgs &a, cudaStream_t s) {
    size_t dyn = 0;
    if (a.mode == PLAN_RD_MIXED || a.mode == PLAN_RD_KV) {
        const cudaError_t attr = once_per_device(0, []() {
            return cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)(4 * kPlanMaxW * 8 + kPlanMaxW * 2));
        });
        if (attr != cudaSuccess) return attr;
        dyn = mixed_plan_smem(L);
    }
    plan_kernel<<<L.B, kPlanThreads, dyn, s>>>(L, C, a);
    return cudaGetLastError();
}

static dim3 work_grid(const LayerDev &L, int max_entries) {
    int gx = max_entries < 1 ? 1 : max_entries;
    if (gx > 256) gx = 256;
    return dim3(gx, L.Hkv * 2, L.B);
}

cudaError_t launch_quantize(const LayerDev &L, const CacheDev &C, int layer, const __nv_bfloat16 *k_ext,
                            const __nv_bfloat16 *v_ext, int64_t ext_len, int max_entries, cudaStream_t s) {
    const int smem = L.w * kHeadDim;
    quantize_kernel<<<work_grid(L, max_entries), 128, smem, s>>>(L, C, layer, k_ext, v_ext, ext_len);
    return cudaGetLastError();
}

cudaError_t launch_promote(const LayerDev &L, const CacheDev &C, int max_entries, cudaStream_t s) {
    (void)C;
    promote_kernel<<<work_grid(L, max_entries), 128, 0, s>>>(L);
    return cudaGetLastError();
}

cudaError_t launch_prefill_copy(const LayerDev &L, const __nv_bfloat16 *k_ext, const __nv_bfloat16 *v_ext,
                                int64_t ext_len, int max_entries, cudaStream_t s) {
    prefill_copy_kernel<<<work_grid(L, max_entries), 128, 0, s>>>(L, k_ext, v_ext, ext_len);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- K channel weights
// "Technische Samenvatting: RDKV", 2.1: w_c = ||Q[:, c]|| ||K[:, c]|| / sqrt(d) per
// (sequence, KV head, channel); the query heads of a KV head pool their columns.
// One cluster of kKwCtas CTAs per (sequence, KV head); CTA r takes the r-th
// contiguous share of the key rows and of the query rows. A thread holds eight
// channels (one 16-byte load per row) and runs over every kKwRowGroups-th row of
// the share; the CTA adds its row groups in order, and rank 0 adds the CTAs'
// sums in rank order from distributed shared memory: fp32 throughout, in a
// fixed order, so that every call gives the same weights.
constexpr int kKwCtas = 8, kKwThreads = 512, kKwRowGroups = kKwThreads / 16;

__device__ __forceinline__ void kw_rows(const __nv_bfloat16 *__restrict__ base, int64_t row_stride, int64_t r0,
                                        int64_t r1, int rg, float (&acc)[8]) {
    int64_t r = r0 + rg;
#pragma unroll 4
    for (; r < r1; r += kKwRowGroups) {
        const uint4 u = __ldcs(reinterpret_cast<const uint4 *>(base + r * row_stride));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xffff0000u);
            acc[2 * j] = fmaf(lo, lo, acc[2 * j]);
            acc[2 * j + 1] = fmaf(hi, hi, acc[2 * j + 1]);
        }
    }
}

__global__ void __cluster_dims__(kKwCtas, 1, 1) __launch_bounds__(kKwThreads)
    k_weights_kernel(LayerDev D, const __nv_bfloat16 *__restrict__ q, int n_q, const __nv_bfloat16 *__restrict__ k,
                     int64_t n_tok, float *out) {
    cg::cluster_group cl = cg::this_cluster();
    const int rank = (int)cl.block_rank();
    const int bh = blockIdx.x / kKwCtas, b = bh / D.Hkv, h = bh % D.Hkv;
    const int tid = threadIdx.x, rg = tid >> 4, c8 = (tid & 15) * 8;   // row group, first channel
    __shared__ float red[2][kKwRowGroups][kHeadDim];
    __shared__ float part[2][kHeadDim];   // this CTA's sums of squares: keys, queries
    float ak[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, aq[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    // key rows t of (b, h): [b][t][h][d]
    kw_rows(k + ((int64_t)b * n_tok * D.Hkv + h) * kHeadDim + c8, (int64_t)D.Hkv * kHeadDim,
            n_tok * rank / kKwCtas, n_tok * (rank + 1) / kKwCtas, rg, ak);
    // query rows (pos, j) of (b, h), pos-major: [b][pos][h G + j][d]
    {
        const int G = D.G;
        const int64_t nr = (int64_t)n_q * G, r0 = nr * rank / kKwCtas, r1 = nr * (rank + 1) / kKwCtas;
        for (int64_t r = r0 + rg; r < r1; r += kKwRowGroups) {
            const int64_t pos = r / G, j = r % G;
            const uint4 u = __ldcs(reinterpret_cast<const uint4 *>(
                q + (((int64_t)b * n_q + pos) * D.Hq + h * G + j) * kHeadDim + c8));
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const float lo = __uint_as_float(w[jj] << 16), hi = __uint_as_float(w[jj] & 0xffff0000u);
                aq[2 * jj] = fmaf(lo, lo, aq[2 * jj]);
                aq[2 * jj + 1] = fmaf(hi, hi, aq[2 * jj + 1]);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        red[0][rg][c8 + j] = ak[j];
        red[1][rg][c8 + j] = aq[j];
    }
    __syncthreads();
    if (tid < 2 * kHeadDim) {
        const int which = tid >> 7, c = tid & (kHeadDim - 1);
        float sum = 0.f;
        for (int i = 0; i < kKwRowGroups; ++i) sum += red[which][i][c];
        part[which][c] = sum;
    }
    cl.sync();   // every CTA's sums are in its shared memory
    if (rank == 0 && tid < kHeadDim) {
        float K2 = 0.f, Q2 = 0.f;
        for (int r = 0; r < kKwCtas; ++r) {
            const float *pr = cl.map_shared_rank(&part[0][0], r);
            K2 += pr[tid];
            Q2 += pr[kHeadDim + tid];
        }
        out[((int64_t)b * D.Hkv + h) * kHeadDim + tid] = sqrtf(Q2) * sqrtf(K2) / sqrtf((float)kHeadDim);
    }
    cl.sync();   // rank 0 has read the others' shared memory
}

cudaError_t launch_k_channel_weights(const LayerDev &L, const __nv_bfloat16 *q, int n_q, const __nv_bfloat16 *k,
                                     int64_t n_tok, float *out, cudaStream_t s) {
    k_weights_kernel<<<L.B * L.Hkv * kKwCtas, kKwThreads, 0, s>>>(L, q, n_q, k, n_tok, out);
    return cudaGetLastError();
}

cudaError_t launch_read_lengths(const LayerDev &L, int32_t *out, cudaStream_t s) {
    read_lengths_kernel<<<1, 32, 0, s>>>(L, out);
    return cudaGetLastError();
}

cudaError_t launch_scores(const LayerDev &L, int n_win, float *out, cudaStream_t s) {
    scores_kernel<<<64, 256, 0, s>>>(L, n_win, out);
    return cudaGetLastError();
}

}  // namespace qevict
