// Split-K single-token GQA decode attention over the three-tier cache, with
// the per-window softmax mass and the cumulative-score update fused in.
//
// Method: "Technische Samenvatting: QEvict" (gist.science 2608.05326),
// "Methodologie: QEvict" (full-precision and INT2 windows stay visible to
// attention, evicted windows do not) and "Kernmechanismen" (cumulative
// scoring, GQA). "Technische Samenvatting: LogQuant" (gist.science
// 2503.19950), Methodologie 3 and 4: evicted tokens leave the softmax
// normalisation, and entries may be visited in any order, which is what lets
// a split walk its full-precision windows first and its INT2 windows after.
//
// Grid (splits, B * Hkv). A CTA owns one (sequence, KV head) and a byte-
// balanced contiguous run of that sequence's window list (full-precision
// windows, then INT2 windows). Each window's K+V for the KV head is one
// contiguous block in HBM and arrives by one cp.async.bulk into a stage of
// a shared-memory ring tracked by mbarriers. The CTA keeps, for each of its G
// query heads, the running max, the running exp-sum and the output
// accumulator, and records every window's own (max, exp-sum). The last CTA
// of a (sequence, KV head) to finish merges the splits (log-sum-exp), writes
// the output, turns the window records into masses and adds their mean over
// the Hq heads into the KV head's partial cumulative score.
#include "qevict_internal.cuh"

namespace qevict {

namespace {

constexpr int kThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitCycles = 4000000000ll;   // about two seconds at GB300 clocks

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on a stage barrier: false after about two seconds.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitCycles) return false;
    }
    return true;
}

// Smallest list entry whose first byte is at or after unit offset u, in the
// concatenated list (n_fp full-precision windows of u_fp bytes, then n_q
// INT2 windows of u_q bytes).
__device__ __forceinline__ int entry_at(int64_t u, int n_fp, int n_q, int64_t u_fp, int64_t u_q) {
    const int64_t fp_total = (int64_t)n_fp * u_fp;
    if (u <= fp_total) return (int)((u + u_fp - 1) / u_fp);
    const int64_t e = n_fp + (u - fp_total + u_q - 1) / u_q;
    return (int)min(e, (int64_t)(n_fp + n_q));
}

template <int G>
__global__ void __launch_bounds__(kThreads) decode_kernel(LayerDev D, CacheDev C, int layer,
                                                           const __nv_bfloat16 *__restrict__ q,
                                                           float *__restrict__ out, float *__restrict__ mass,
                                                           int accumulate, int splits, int nst,
                                                           int stage_bytes) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int w = D.w;
    uint8_t *stages = smem;
    float *q_s = reinterpret_cast<float *>(smem + (size_t)nst * stage_bytes);   // [G][d]
    float *p_s = q_s + G * kHeadDim;                                             // [G][w]
    float *run_m = p_s + G * w;                                                  // [G]
    float *run_l = run_m + kMaxG;
    float *s_alpha = run_l + kMaxG;
    float *s_M = s_alpha + kMaxG;
    float *s_il = s_M + kMaxG;
    uint64_t *bars = reinterpret_cast<uint64_t *>(s_il + kMaxG);                // [nst]
    __shared__ int s_flag;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x;
    const int bk = blockIdx.y;
    const int b = bk / D.Hkv, kvh = bk % D.Hkv;
    const int Hq = D.Hq;
    const int64_t wb = (int64_t)b * D.Wmax;
    const int64_t length = D.ctr[b * kCtrN + CTR_LEN];
    const int n_win = (int)((length + w - 1) / w);

    // query, pre-scaled so that logits are in the log2 domain
    const float qscale = kLog2e * rsqrtf((float)kHeadDim);
    for (int i = tid; i < G * kHeadDim; i += kThreads) {
        const int g = i / kHeadDim, j = i % kHeadDim;
        q_s[i] = __bfloat162float(q[((int64_t)b * Hq + kvh * G + g) * kHeadDim + j]) * qscale;
    }
    if (tid < kMaxG) {
        run_m[tid] = -INFINITY;
        run_l[tid] = 0.f;
    }

    // this split's run of the window list
    const int n_fp = D.ctr[b * kCtrN + CTR_NFP];
    const int n_q = D.ctr[b * kCtrN + CTR_NQ];
    const int64_t u_fp = (int64_t)w * kHeadDim * 4;          // K + V bf16 for one KV head
    const int64_t u_q = 2 * lg_part_bytes(w);                // K + V codes + meta
    const int64_t U = n_fp * u_fp + n_q * u_q;
    const int e0 = entry_at(U * split / splits, n_fp, n_q, u_fp, u_q);
    const int e1 = entry_at(U * (split + 1) / splits, n_fp, n_q, u_fp, u_q);

    if (tid == 0) {
        s_flag = 0;
        for (int i = 0; i < nst; ++i) mbar_init(&bars[i], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    auto issue = [&](int e, int st) {
        const bool fp = e < n_fp;
        const int2 ent = fp ? D.fp_list[b * D.CF + e] : D.q_list[b * D.CQ + (e - n_fp)];
        const uint8_t *src;
        uint32_t bytes;
        if (fp) {
            src = D.fp_pool + (int64_t)ent.y * D.fp_slot_bytes + (int64_t)kvh * u_fp;
            bytes = (uint32_t)u_fp;
        } else {
            src = D.lg_pool + (int64_t)ent.y * D.lg_slot_bytes + (int64_t)kvh * u_q;
            bytes = (uint32_t)u_q;
        }
        mbar_expect_tx(&bars[st], bytes);
        bulk_g2s(stages + (size_t)st * stage_bytes, src, bytes, &bars[st]);
    };
    int issued_end = e0;   // thread 0: entries [e0, issued_end) have been issued
    if (tid == 0) {
        for (int i = 0; i < nst && e0 + i < e1; ++i) issue(e0 + i, i);
        issued_end = min(e1, e0 + nst);
    }

    float acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = 0.f;

    for (int e = e0; e < e1; ++e) {
        const int it = e - e0;
        const int st = it % nst;
        const uint32_t parity = (uint32_t)((it / nst) & 1);
        const bool ok = mbar_wait(&bars[st], parity);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                set_status(C, QEVICT_ERR_TIMEOUT, layer, b, e);
                // let the copies still in flight land before the CTA moves on
                for (int r = e; r < issued_end; ++r)
                    (void)mbar_wait(&bars[(r - e0) % nst], (uint32_t)(((r - e0) / nst) & 1));
            }
            break;
        }
        const bool fp = e < n_fp;
        const int2 ent = fp ? D.fp_list[b * D.CF + e] : D.q_list[b * D.CQ + (e - n_fp)];
        const int wi = ent.x;
        const int ntok = (wi == n_win - 1) ? (int)(length - (int64_t)wi * w) : w;
        const uint8_t *sb = stages + (size_t)st * stage_bytes;

        // ---- logits: warp per token, lane per 4 channels
        for (int t = warp; t < w; t += kThreads / 32) {
            float k4[4];
            if (fp) {
                const uint2 u = reinterpret_cast<const uint2 *>(sb + (size_t)t * kHeadDim * 2)[lane];
                const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
                const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
                k4[0] = a.x; k4[1] = a.y; k4[2] = c.x; k4[3] = c.y;
            } else {
                const uint32_t byte = sb[(size_t)t * (kHeadDim / 4) + lane];
                const __half2 m2 = reinterpret_cast<const __half2 *>(sb + lg_codes_bytes(w))[t * kGroups + lane / 8];
                const float s = __low2float(m2), mn = __high2float(m2);
#pragma unroll
                for (int i = 0; i < 4; ++i) k4[i] = fmaf((float)((byte >> (2 * i)) & 3u), s, mn);
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float4 qv = reinterpret_cast<const float4 *>(q_s + g * kHeadDim)[lane];
                float dot = qv.x * k4[0] + qv.y * k4[1] + qv.z * k4[2] + qv.w * k4[3];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
                if (lane == 0) p_s[g * w + t] = t < ntok ? dot : -INFINITY;
            }
        }
        __syncthreads();

        // ---- window statistics and probabilities (warp per head)
        for (int g = warp; g < G; g += kThreads / 32) {
            float mw = -INFINITY;
            for (int t = lane; t < ntok; t += 32) mw = fmaxf(mw, p_s[g * w + t]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, o));
            const float m_old = run_m[g];
            const float m_new = fmaxf(m_old, mw);
            const float beta = exp2f(mw - m_new);
            float es = 0.f;
            for (int t = lane; t < w; t += 32) {
                const float ex = t < ntok ? exp2f(p_s[g * w + t] - mw) : 0.f;
                es += ex;
                p_s[g * w + t] = ex * beta;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) es += __shfl_xor_sync(0xffffffffu, es, o);
            if (lane == 0) {
                const float alpha = m_old == -INFINITY ? 0.f : exp2f(m_old - m_new);
                run_l[g] = run_l[g] * alpha + es * beta;
                run_m[g] = m_new;
                s_alpha[g] = alpha;
                D.wstat[((int64_t)b * Hq + kvh * G + g) * D.Wmax + wi] = make_float2(mw, es);
            }
        }
        __syncthreads();

        // ---- P.V: thread per channel
        {
            const int j = tid;
#pragma unroll
            for (int g = 0; g < G; ++g) acc[g] *= s_alpha[g];
            if (fp) {
                const __nv_bfloat16 *vb = reinterpret_cast<const __nv_bfloat16 *>(sb) + (size_t)w * kHeadDim;
                for (int t = 0; t < ntok; ++t) {
                    const float vv = __bfloat162float(vb[(size_t)t * kHeadDim + j]);
#pragma unroll
                    for (int g = 0; g < G; ++g) acc[g] = fmaf(p_s[g * w + t], vv, acc[g]);
                }
            } else {
                const uint8_t *vpart = sb + lg_part_bytes(w);
                const uint32_t *vw = reinterpret_cast<const uint32_t *>(vpart);
                const __half2 *vm = reinterpret_cast<const __half2 *>(vpart + lg_codes_bytes(w));
                for (int t = 0; t < ntok; ++t) {
                    const uint32_t c = (vw[(t / kVTile) * kHeadDim + j] >> (2 * (t % kVTile))) & 3u;
                    const __half2 m2 = vm[t * kGroups + j / kGroup];
                    const float vv = fmaf((float)c, __low2float(m2), __high2float(m2));
#pragma unroll
                    for (int g = 0; g < G; ++g) acc[g] = fmaf(p_s[g * w + t], vv, acc[g]);
                }
            }
        }
        __syncthreads();
        if (tid == 0 && e + nst < e1) {
            issue(e + nst, st);
            issued_end = e + nst + 1;
        }
    }

    // ---- split partials
    float *part = D.part + (((int64_t)b * D.Hkv + kvh) * kMaxSplits + split) * G * (2 + kHeadDim);
#pragma unroll
    for (int g = 0; g < G; ++g) part[g * (2 + kHeadDim) + 2 + tid] = acc[g];
    if (tid < G) {
        part[tid * (2 + kHeadDim)] = run_m[tid];
        part[tid * (2 + kHeadDim) + 1] = run_l[tid];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(&D.arrive[bk], 1u);
        s_flag = prev == (unsigned)(splits - 1);
    }
    __syncthreads();
    if (!s_flag) return;
    __threadfence();

    // ---- last CTA: log-sum-exp merge of the splits
    const float *pb = D.part + ((int64_t)b * D.Hkv + kvh) * kMaxSplits * G * (2 + kHeadDim);
    if (tid < G) {
        float M = -INFINITY;
        for (int s = 0; s < splits; ++s) M = fmaxf(M, __ldcg(pb + ((int64_t)s * G + tid) * (2 + kHeadDim)));
        float l = 0.f;
        if (M != -INFINITY) {
            for (int s = 0; s < splits; ++s) {
                const float ms = __ldcg(pb + ((int64_t)s * G + tid) * (2 + kHeadDim));
                const float ls = __ldcg(pb + ((int64_t)s * G + tid) * (2 + kHeadDim) + 1);
                if (ms != -INFINITY) l += ls * exp2f(ms - M);
            }
        }
        s_M[tid] = M;
        s_il[tid] = l > 0.f ? 1.f / l : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float o = 0.f;
        const float M = s_M[g];
        if (M != -INFINITY) {
            for (int s = 0; s < splits; ++s) {
                const float ms = __ldcg(pb + ((int64_t)s * G + g) * (2 + kHeadDim));
                if (ms == -INFINITY) continue;
                o = fmaf(__ldcg(pb + ((int64_t)s * G + g) * (2 + kHeadDim) + 2 + tid), exp2f(ms - M), o);
            }
        }
        out[((int64_t)b * Hq + kvh * G + g) * kHeadDim + tid] = o * s_il[g];
    }
    // masses and the cumulative score
    const float inv_hq = 1.f / (float)Hq;
    for (int wi = tid; wi < n_win; wi += kThreads) {
        const bool live = D.tier[wb + wi] != QEVICT_TIER_E;
        float sum = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float m = 0.f;
            if (live && s_M[g] != -INFINITY) {
                const float2 ws = __ldcg(&D.wstat[((int64_t)b * Hq + kvh * G + g) * D.Wmax + wi]);
                m = ws.y * exp2f(ws.x - s_M[g]) * s_il[g];
            }
            if (mass) mass[((int64_t)b * Hq + kvh * G + g) * n_win + wi] = m;
            sum += m;
        }
        if (accumulate) D.score_part[((int64_t)b * D.Hkv + kvh) * D.Wmax + wi] += sum * inv_hq;
    }
    if (tid == 0) D.arrive[bk] = 0u;
}

}  // namespace

int decode_smem_bytes(int w, int G) {
    (void)G;
    const int stage = w * kHeadDim * 4;
    const int extra = kMaxG * kHeadDim * 4 + kMaxG * w * 4 + 5 * kMaxG * 4 + 8 * 8 + 128;
    int nst = (200 * 1024 - extra) / stage;
    if (nst > 4) nst = 4;
    if (nst < 2) nst = 2;
    return nst * stage + extra;
}

cudaError_t launch_decode(const LayerDev &L, const CacheDev &C, int layer, const __nv_bfloat16 *q, float *out,
                          float *mass, int accumulate, int splits, cudaStream_t s) {
    const int stage = L.w * kHeadDim * 4;
    const int smem = decode_smem_bytes(L.w, L.G);
    const int extra = kMaxG * kHeadDim * 4 + kMaxG * L.w * 4 + 5 * kMaxG * 4 + 8 * 8 + 128;
    const int nst = (smem - extra) / stage;
    dim3 grid(splits, L.B * L.Hkv);
#define QV_CASE(GG)                                                                                    \
    case GG: {                                                                                         \
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<GG>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                             smem);                                                    \
        if (e != cudaSuccess) return e;                                                                \
        decode_kernel<GG><<<grid, kThreads, smem, s>>>(L, C, layer, q, out, mass, accumulate, splits, nst,    \
                                                       stage);                            \
        break;                                                                                         \
    }
    switch (L.G) {
        QV_CASE(1)
        QV_CASE(2)
        QV_CASE(3)
        QV_CASE(4)
        QV_CASE(5)
        QV_CASE(6)
        QV_CASE(7)
        QV_CASE(8)
        default:
            return cudaErrorInvalidValue;
    }
#undef QV_CASE
    return cudaGetLastError();
}

}  // namespace qevict
