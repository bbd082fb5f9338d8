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

__device__ __forceinline__ void fmm_add(FmmStat &st, float x, bool evicted) {
    if (x > st.m) {
        const float f = exp2f(st.m - x);
        st.la *= f;
        st.le *= f;
        st.m = x;
    }
    const float e = exp2f(x - st.m);
    st.la += e;
    if (evicted) st.le += e;
}

// One CTA per (split of the token range, sequence and KV head). A warp takes
// chunks of 16 tokens and computes their logits on the tensor cores
// (mma.sync m16n8k16, bf16 operands, fp32 sums): tokens are the M rows, the
// query heads of the group the N columns (padded to 8), channels the K
// dimension in 8 steps of 16. Lane (g, c) = (lane / 4, lane % 4) loads, for
// tokens g and g + 8, the 16-byte pieces at bytes 16 c + 64 i (i = 0..3) of
// the token's 256-byte key row, so the 32 lanes of one load read 8 whole
// 64-byte runs. Inside a 16-channel step the channel order is permuted the
// same way for K and q (lane c's k indices 2c, 2c+1, 2c+8, 2c+9 are its 4
// consecutive channels), which leaves every dot product unchanged and lets
// the loaded words serve as the A fragment as they are. The next chunk's
// keys and tiers are loaded before the current chunk's arithmetic. Each lane
// keeps a running (max, sums) for heads 2c and 2c + 1.
template <int G>
__global__ void __launch_bounds__(kFmmWarps * 32) fmm_partial_kernel(const LayerDev D, const __nv_bfloat16 *q,
                                                                     const __nv_bfloat16 *k_full, int L,
                                                                     float *part, int splits) {
    const int split = blockIdx.x, bk = blockIdx.y;
    const int b = bk / D.Hkv, kvh = bk % D.Hkv;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    const float scale = kLog2eF * rsqrtf((float)kHeadDim);

    // B fragments (q^T): step kk uses channels 8c + 32 (kk / 2) + 4 (kk % 2) + 0..3 of head g
    uint32_t qb[8][2];
    {
        uint4 r[4] = {};
        if (g < G) {
            const uint4 *qp = reinterpret_cast<const uint4 *>(q + ((int64_t)b * D.Hq + kvh * G + g) * kHeadDim);
#pragma unroll
            for (int i = 0; i < 4; ++i) r[i] = qp[c + 4 * i];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            qb[2 * i][0] = r[i].x;
            qb[2 * i][1] = r[i].y;
            qb[2 * i + 1][0] = r[i].z;
            qb[2 * i + 1][1] = r[i].w;
        }
    }
    FmmStat st[2] = {{-INFINITY, 0.f, 0.f}, {-INFINITY, 0.f, 0.f}};

    const int t0 = (int)((int64_t)L * split / splits), t1 = (int)((int64_t)L * (split + 1) / splits);
    const int64_t row = (int64_t)D.Hkv * kHeadDim;   // elements between consecutive tokens
    const uint4 *kb = reinterpret_cast<const uint4 *>(k_full + ((int64_t)b * L * D.Hkv + kvh) * kHeadDim) + c;
    const uint8_t *tier = D.tier + (int64_t)b * D.Wmax;
    // r[h][i]: token g + 8 h, piece i; ev[h]: that token is evicted
    auto load_chunk = [&](int c0, uint4 (&r)[2][4], bool (&ev)[2]) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int t = c0 + g + 8 * h;
            const bool in = t < t1;
            const uint4 *p = kb + (int64_t)t * (row / 8);
#pragma unroll
            for (int i = 0; i < 4; ++i) r[h][i] = in ? __ldg(p + 4 * i) : make_uint4(0, 0, 0, 0);
            ev[h] = in && __ldg(tier + t / D.w) == QEVICT_TIER_E;
        }
    };
    uint4 cur[2][4], nxt[2][4];
    bool ecur[2], enxt[2];
    int c0 = t0 + warp * 16;
    constexpr int stride = kFmmWarps * 16;
    if (c0 < t1) load_chunk(c0, cur, ecur);
    for (; c0 < t1; c0 += stride) {
        if (c0 + stride < t1) load_chunk(c0 + stride, nxt, enxt);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // A fragment: (token g, k 2c..2c+1), (token g+8, same), (token g, k 2c+8..9), (token g+8, same)
            mma_bf16(acc, make_uint4(cur[0][i].x, cur[1][i].x, cur[0][i].y, cur[1][i].y), qb[2 * i][0],
                     qb[2 * i][1]);
            mma_bf16(acc, make_uint4(cur[0][i].z, cur[1][i].z, cur[0][i].w, cur[1][i].w), qb[2 * i + 1][0],
                     qb[2 * i + 1][1]);
        }
        // acc: (token g, head 2c), (token g, head 2c+1), (token g+8, head 2c), (token g+8, head 2c+1)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (c0 + g + 8 * h < t1) {
                if (2 * c < G) fmm_add(st[0], acc[2 * h] * scale, ecur[h]);
                if (2 * c + 1 < G) fmm_add(st[1], acc[2 * h + 1] * scale, ecur[h]);
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            ecur[h] = enxt[h];
#pragma unroll
            for (int i = 0; i < 4; ++i) cur[h][i] = nxt[h][i];
        }
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
    }
}

// One warp per (sequence, query head): lanes take the splits in turn, then
// the lanes' statistics are merged across the warp.
__global__ void fmm_merge_kernel(const LayerDev D, const float *part, int splits, float *fmm) {
    const int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (i >= D.B * D.Hq) return;
    const int b = i / D.Hq, h = i % D.Hq, kvh = h / D.G, hh = h % D.G;
    const int bk = b * D.Hkv + kvh;
    FmmStat acc{-INFINITY, 0.f, 0.f};
    for (int s = lane; s < splits; s += 32) {
        const float *o = part + (((int64_t)bk * splits + s) * D.G + hh) * 3;
        acc = fmm_merge(acc, FmmStat{o[0], o[1], o[2]});
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const FmmStat p{__shfl_xor_sync(0xffffffffu, acc.m, o), __shfl_xor_sync(0xffffffffu, acc.la, o),
                        __shfl_xor_sync(0xffffffffu, acc.le, o)};
        acc = fmm_merge(acc, p);
    }
    if (lane == 0) fmm[i] = acc.la > 0.f ? acc.le / acc.la : 0.f;
}

}  // namespace

cudaError_t launch_future_missed_mass(const LayerDev &L, const CacheDev &C, const DecodeScratch &S, int layer,
                                      const __nv_bfloat16 *q, const __nv_bfloat16 *k_full, int n_tokens, float *fmm,
                                      int num_sms, cudaStream_t s) {
    (void)C;
    (void)layer;
    const int pairs = L.B * L.Hkv;
    // Partials (3 floats per split and query head) go to the window-statistics
    // area of the decode scratch, which holds 2 * Wmax floats per query head
    // and carries nothing from one decode launch to the next. (The partial
    // output area is not used: its words carry arrival tags.)
    float *part = reinterpret_cast<float *>(S.wstat);
    // as many CTAs as fit the GPU at once, spread over the (sequence, KV head) pairs
    auto grid_for = [&](const void *fn) {
        static int per_sm[kMaxG + 1] = {};
        if (!per_sm[L.G] && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm[L.G], fn, kFmmWarps * 32, 0) !=
                                cudaSuccess)
            per_sm[L.G] = 1;
        int splits = (max(1, per_sm[L.G]) * num_sms + pairs - 1) / pairs;
        return max(1, min(splits, min(256, 2 * L.Wmax / 3)));
    };
    int splits = 1;
    switch (L.G) {
#define QV_CASE(GG)                                                                                          \
    case GG:                                                                                                 \
        splits = grid_for((const void *)fmm_partial_kernel<GG>);                                             \
        fmm_partial_kernel<GG><<<dim3(splits, pairs), kFmmWarps * 32, 0, s>>>(L, q, k_full, n_tokens, part,  \
                                                                              splits);                       \
        break;
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
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int n = L.B * L.Hq;
    fmm_merge_kernel<<<(n + 3) / 4, 128, 0, s>>>(L, part, splits, fmm);
    return cudaGetLastError();
}

}  // namespace qevict
