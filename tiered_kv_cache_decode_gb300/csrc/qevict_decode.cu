// Split-K single-token GQA decode attention over the three-tier cache, with
// the per-window softmax mass, the cumulative-score update and (optionally)
// the append of this step's token fused in.
//
// Method: "Technische Samenvatting: QEvict" (gist.science 2608.05326),
// "Methodologie: QEvict" (full-precision and INT2 windows stay visible to
// attention, evicted windows do not) and "Kernmechanismen" (cumulative
// scoring, GQA). "Technische Samenvatting: LogQuant" (gist.science
// 2503.19950), Methodologie 3 and 4: evicted tokens leave the softmax
// normalisation, and cache entries may be visited in any order.
//
// Layout of the work. Grid (splits, B * Hkv); a CTA owns one (sequence, KV
// head) and a cost-balanced contiguous run of that sequence's window list
// (full-precision windows first, then INT2 windows). Its windows are cut
// into 16-token units that its four warps take round-robin. Every warp feeds
// itself: lane 0 keeps three shared-memory stages in flight (a full-precision
// unit is one 4-D TMA tile load of its K and V, 128-byte swizzled; a stage
// takes up to five INT2 units, one bulk copy each of the unit's codes and
// fp16 scale/min) and refills a stage as soon as it has consumed it.
//
// Per unit a warp computes the GQA query group's logits and P.V on the
// tensor cores (mma.sync m16n8k16, bf16 operands, fp32 accumulation):
//  - QK: S[head][token] = Q[head][:] . K[token][:]; the G query heads are the
//    M rows (padded to 16), 8 tokens per N tile. INT2 codes 0..3 are exact in
//    bf16 and built in registers (code | 0x4300 is 128 + code; minus 128),
//    one accumulator per group of 32 channels, then
//    logit = sum_g scale_g * acc_g + min_g * sum(q over group g): the exact
//    reconstruction min + code * scale, never rounded.
//  - PV: O^T[channel][head] += V^T[channel][token] . P^T[token][head]; P is
//    split into bf16 hi + lo parts (two MMAs) so it keeps ~16 bits; for INT2
//    the scale folds into P per group and the min term is a CUDA-core sum.
//    (An fp16 P * scale with one MMA keeps only 11 bits: heavy-tailed V
//    groups then miss a 2e-3 absolute bound.)
//  The token order inside an INT2 unit is permuted (pairs t, t+8 share a
//  32-bit code word) and the same permutation is used on both sides of each
//  product, which leaves every sum unchanged.
// The last CTA of a (sequence, KV head) merges the splits by log-sum-exp,
// adds this step's token when one is given, writes the output, turns the
// per-window (max, exp-sum) records into masses and adds their mean over the
// Hq heads into the KV head's partial cumulative score; the last of the
// sequence's KV heads then opens the new window / advances the length.
//
// With programmatic dependent launch the kernel starts loading cache units
// before the previous kernel in the stream has finished and waits for it
// only before it reads the query (griddepcontrol.wait); the host enables
// this only when that previous kernel did not change this layer's cache.
#include "qevict_internal.cuh"

namespace qevict {

namespace {

constexpr int kWarps = 12;                // warps per CTA (one CTA per SM)
constexpr int kThreads = kWarps * 32;
constexpr int kTailThreads = (kWarps - 1) * 32;   // threads of the split merge (the last warp appends)
// shared-memory offsets used after the main loop (inside the free rings)
constexpr int kHeadOff = 54 * 1024;    // per-head merge results, per-split weights, new token's V row
constexpr int kRedOff = 58 * 1024;     // [<= 288] float4 weighted split partials of this CTA's output slice
constexpr int kStages = 2;                // shared-memory stages per warp
constexpr int kStage = 8192;              // bytes per stage
constexpr int kRing = kStages * kStage;   // bytes per warp
constexpr int kFPUnit = 8192;             // 16 tokens x (K, V) x 256 B: one per stage
constexpr int kQUnit = 1536;              // 16 tokens: K codes 512, K meta 256, V codes 512, V meta 256
constexpr int kQPerStage = kStage / kQUnit;   // INT2 units batched into one stage (5)
constexpr int kEntTab = 1024;             // window-list entries of a split cached in shared memory
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.f;              // log2 headroom before the running max moves
constexpr long long kWaitCycles = 4000000000ll;   // about two seconds at GB300 clocks

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// try_wait suspends the thread until the phase completes or about 20 us pass
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
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}
// L2 policy for data read once per launch: evicted first, so that it does not
// push the kernel's code, tables and scratch out of L2
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tma_4d(uint32_t dst, const CUtensorMap *map, int x, int y, int z, int u,
                                       uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(u), "r"(bar), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                    uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D = A B + C with C from separate registers: {c0, c0, c1, c1}
__device__ __forceinline__ void mma_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                      uint32_t b1, float c0, float c1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %10, %11, %11};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1));
}
// barrier among the merge warps of the last CTA (named barrier 1)
__device__ __forceinline__ void tail_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kTailThreads) : "memory"); }
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
// Two 2-bit codes (bits 1:0 and 17:16 of x) as an exact bf16 pair.
__device__ __forceinline__ uint32_t codes2(uint32_t x) {
    uint32_t r = (x & 0x00030003u) | 0x43004300u;     // bf16 128 + code in each half
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&r);
    v = __hsub2(v, __floats2bfloat162_rn(128.f, 128.f));
    return *reinterpret_cast<uint32_t *>(&v);
}
// K codes of a QK k-step as bf16 pairs with the offset kept: bits 1:0 and
// 17:16 give 128 + code, bits 3:2 and 19:18 give 128 + 4 code (both exact).
// The query values that meet the second pair are stored divided by 4, and
// the offsets' contribution is taken out through the accumulator's start value.
__device__ __forceinline__ uint32_t kcodes_lo(uint32_t x) { return (x & 0x00030003u) | 0x43004300u; }
__device__ __forceinline__ uint32_t kcodes_hi(uint32_t x) { return (x & 0x000C000Cu) | 0x43004300u; }
// The same for 4-bit codes c = c0 + 4 c1 held in two 2-bit planes (x0: c0, x1:
// c1, at the same bit positions): 128 + c and 128 + 4 c, exact in bf16.
__device__ __forceinline__ uint32_t kcodes4_lo(uint32_t x0, uint32_t x1) {
    return (x0 & 0x00030003u) | ((x1 & 0x00030003u) << 2) | 0x43004300u;
}
__device__ __forceinline__ uint32_t kcodes4_hi(uint32_t x0, uint32_t x1) {
    return (x0 & 0x000C000Cu) | ((x1 & 0x000C000Cu) << 2) | 0x43004300u;
}
// Two 4-bit codes (bits 1:0 and 17:16 of each plane word) as an exact bf16 pair.
__device__ __forceinline__ uint32_t codes4(uint32_t x0, uint32_t x1) {
    uint32_t r = kcodes4_lo(x0, x1);
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&r);
    v = __hsub2(v, __floats2bfloat162_rn(128.f, 128.f));
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
// hi = x truncated to bf16 (its top 16 bits), lo = bf16_rn(x - hi) for a pair:
// hi + lo carries x to within 2^-16 relative.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const uint32_t u0 = __float_as_uint(x0), u1 = __float_as_uint(x1);
    hi = __byte_perm(u0, u1, 0x7632);
    lo = pack2(x0 - __uint_as_float(u0 & 0xffff0000u), x1 - __uint_as_float(u1 & 0xffff0000u));
}
__device__ __forceinline__ float2 h2f(uint32_t u) {
    const __half2 h = *reinterpret_cast<const __half2 *>(&u);
    return __half22float2(h);
}
__device__ __forceinline__ uint32_t pick(const uint4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// 2^x (PTX ex2.approx; results below 2^-126 flush to zero)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// (max, exp-sum relative to max) pairs
__device__ __forceinline__ float2 stat_merge(float2 a, float2 b) {
    if (a.y <= 0.f) return b;
    if (b.y <= 0.f) return a;
    const float m = fmaxf(a.x, b.x);
    return make_float2(m, a.y * ex2(a.x - m) + b.y * ex2(b.x - m));
}

// A split's share of the window list: full-precision entries [f0, f1) and
// INT2 entries [q0, q1) (indices within each tier's list). Every split gets a
// proportional share of each tier, so memory-bound and ALU-bound work mix
// evenly over the CTAs.
struct Range {
    int f0, f1, q0, q1;
};

__device__ __forceinline__ Range split_range(int split, int splits, int n_fp, int n_q) {
    return Range{(int)((int64_t)n_fp * split / splits), (int)((int64_t)n_fp * (split + 1) / splits),
                 (int)((int64_t)n_q * split / splits), (int)((int64_t)n_q * (split + 1) / splits)};
}

// kWide: the cache may hold INT4 / INT8 windows (2 or 4 code planes); the
// instantiation without it is the INT2 / full-precision kernel as such.
template <int G, bool kWide>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const LayerDev D, const CacheDev C, const DecodeScratch S, const __grid_constant__ CUtensorMap tmap,
                  int layer, const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *knew,
                  const __nv_bfloat16 *vnew, float *__restrict__ out, float *__restrict__ mass, int accumulate,
                  int splits) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 128-byte-swizzled TMA tiles need 1024-byte aligned destinations
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    int2 *s_ent = reinterpret_cast<int2 *>(smem + kWarps * kRing);   // this split's {window, slot} list
    // query A fragments per lane: [path (0 natural, 1 INT2 channel order)][k-step][lane] {a0, a2}
    uint2 *s_qf = reinterpret_cast<uint2 *>(smem + kWarps * kRing + kEntTab * 8);
    __shared__ uint64_t bars[kWarps][kStages];
    __shared__ uint32_t s_gen;                               // split-record generation of this launch
    __shared__ int st_n[kWarps][kStages];                    // units in a stage
    __shared__ int st_fp[kWarps][kStages];                   // 1: a full-precision unit
    __shared__ int st_p[kWarps][kStages];                    // code planes of a quantised stage (kWide)
    __shared__ int st_wi[kWarps][kStages][kQPerStage];       // window of each unit
    __shared__ int st_j[kWarps][kStages][kQPerStage];        // 16-token unit index inside the window
    __shared__ int st_nt[kWarps][kStages][kQPerStage];       // tokens in the unit
    __shared__ int st_emit[kWarps][kStages][kQPerStage];     // window statistics after the unit: 1 whole, 2 partial
    __shared__ int pt_win[kWarps][2];                        // windows this warp saw only part of
    __shared__ float2 pt_st[kWarps][2][8];                   // their (max, exp-sum) per head

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int split = blockIdx.x, bk = blockIdx.y;
    const int Hkv = D.Hkv, Hq = D.Hq, w = D.w, mu = w / 16;
    const int b = bk / Hkv, kvh = bk % Hkv;
    const int64_t wb = (int64_t)b * D.Wmax;
    const int32_t *ctr = D.ctr + b * kCtrN;
    const int64_t length = ctr[CTR_LEN];
    if (knew != nullptr && length >= D.max_context) {   // replayed past the end of the tables
        if (tid == 0 && split == 0) set_status(C, QEVICT_ERR_INVALID_ARG, layer, b, (int)length);
        knew = nullptr;
        vnew = nullptr;
    }
    const int n_win = (int)((length + w - 1) / w);
    const int n_fp = ctr[CTR_NFP], n_q = ctr[CTR_NQ];
    const Range R = split_range(split, splits, n_fp, n_q);
    const int nfw = R.f1 - R.f0;                       // full-precision windows of this split
    const int nwin = nfw + (R.q1 - R.q0);              // windows of this split
    const uint32_t ring_s = smem_u32(smem + warp * kRing);

    // ---- this split's windows: local index i (full-precision first, then INT2)
    auto lentry = [&](int i) -> int2 {
        return i < nfw ? D.fp_list[b * D.CF + R.f0 + i] : D.q_list[b * D.CQ + R.q0 + (i - nfw)];
    };
    for (int i = tid; i < min(nwin, kEntTab); i += kThreads) s_ent[i] = lentry(i);
    if (lane == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(smem_u32(&bars[warp][i]), 1);
        pt_win[warp][0] = pt_win[warp][1] = -1;
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();
    auto ent = [&](int i) -> int2 { return i < kEntTab ? s_ent[i] : lentry(i); };
    auto ntok_of = [&](int wi) -> int { return (wi == n_win - 1) ? (int)(length - (int64_t)wi * w) : w; };

    // ---- issue bookkeeping (all lanes run it; lane 0 issues the copies). The
    // split's windows are cut into 16-token units (w / 16 per window; the open
    // window's units past its last token are skipped) and each warp takes a
    // contiguous range of them. A stage holds one full-precision unit, or up
    // to five INT2 tiles (one bulk copy per window's run of tiles). A window
    // whose units all lie in this warp's range gets its statistics written
    // after its last unit; a window cut by a range boundary leaves a partial
    // entry, merged with its neighbour's after the loop.
    const uint64_t l2_stream = evict_first_policy();
    const int n_units = nwin * mu;
    // unit -> (window, unit in window): a shift when mu is a power of two
    const bool mu_pow2 = (mu & (mu - 1)) == 0;
    const int lmu = 31 - __clz(mu);
    auto win_of = [&](int u) -> int { return mu_pow2 ? u >> lmu : u / mu; };
    const int u_beg = (int)((int64_t)n_units * warp / kWarps);
    const int u_end = (int)((int64_t)n_units * (warp + 1) / kWarps);
    int iu = u_beg;                  // next unit to issue
    int issued = 0, consumed = 0;    // stages issued / consumed
    auto try_issue = [&]() {
        while (iu < u_end && issued - consumed < kStages) {
            const int li = win_of(iu), j = iu - li * mu;
            const int st = issued % kStages;
            const uint32_t bar = smem_u32(&bars[warp][st]);
            const uint32_t dst = ring_s + st * kStage;
            if (li < nfw) {
                const int2 en = ent(li);
                const int nt = ntok_of(en.x);
                const int nu = (nt + 15) >> 4;   // units that hold tokens
                if (j >= nu) {                   // past the open window's last token
                    iu = (li + 1) * mu;
                    continue;
                }
                if (lane == 0) {
                    const bool whole = li * mu >= u_beg && li * mu + nu <= u_end;
                    st_n[warp][st] = 1;
                    st_fp[warp][st] = 1;
                    st_wi[warp][st][0] = en.x;
                    st_j[warp][st][0] = j;
                    st_nt[warp][st][0] = min(16, nt - 16 * j);
                    st_emit[warp][st][0] = (j == nu - 1 || iu + 1 == u_end) ? (whole ? 1 : 2) : 0;
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_expect_tx(bar, (uint32_t)kFPUnit);
                    tma_4d(dst, &tmap, 0, 16 * j, 0, en.y * Hkv + kvh, bar, l2_stream);
                }
                ++iu;
            } else {
                // quantised windows are always full (mu tiles); with kWide a stage
                // holds the tiles of one width only (2560 / 4608 B for INT4 / INT8)
                int P = 1, tb = kQUnit, n = min(kQPerStage, u_end - iu);
                if (kWide) {
                    P = 1 << (ent(win_of(iu)).y >> kSlotBits);
                    tb = qtile_bytes(P);
                    n = 0;
                    for (int iu2 = iu; iu2 < u_end && n < kStage / tb;) {
                        const int lq = win_of(iu2);
                        if ((1 << (ent(lq).y >> kSlotBits)) != P) break;
                        const int run = min(min(mu - (iu2 - lq * mu), kStage / tb - n), u_end - iu2);
                        n += run;
                        iu2 += run;
                    }
                }
                if (lane == 0) {
                    st_n[warp][st] = n;
                    st_fp[warp][st] = 0;
                    if (kWide) st_p[warp][st] = P;
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_expect_tx(bar, (uint32_t)(n * tb));
                }
                int done = 0;
                while (done < n) {
                    const int lq = win_of(iu), jq = iu - lq * mu;
                    const int2 en = ent(lq);
                    const int slot = kWide ? (en.y & ((1 << kSlotBits) - 1)) : en.y;
                    const int run = min(mu - jq, n - done);
                    if (lane == 0) {
                        const bool whole = lq * mu >= u_beg && (lq + 1) * mu <= u_end;
                        for (int r = 0; r < run; ++r) {
                            st_wi[warp][st][done + r] = en.x;
                            st_j[warp][st][done + r] = jq + r;
                            st_nt[warp][st][done + r] = 16;
                            st_emit[warp][st][done + r] =
                                (jq + r == mu - 1 || iu + r + 1 == u_end) ? (whole ? 1 : 2) : 0;
                        }
                        bulk_g2s(dst + done * tb,
                                 D.lg_pool + (int64_t)slot * D.lg_slot_bytes +
                                     (kWide ? lg_tile_off(kvh, w, jq, P) : lg_tile_off(kvh, w, jq)),
                                 (uint32_t)(run * tb), bar, l2_stream);
                    }
                    done += run;
                    iu += run;
                }
            }
            ++issued;
        }
    };
    try_issue();   // cache data only: safe before the dependency wait

    // ---- wait for the previous kernel, then let the next one start
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0) s_gen = *(volatile const uint32_t *)(S.bar + 2 * bk + 1);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ---- query fragments (A operand: G heads as rows, rest zero)
    const uint32_t *qw =
        reinterpret_cast<const uint32_t *>(q + ((int64_t)b * Hq + kvh * G + (g < G ? g : 0)) * kHeadDim);
    float qsum[kGroups] = {0.f, 0.f, 0.f, 0.f};
    float qbias[kGroups] = {0.f, 0.f, 0.f, 0.f};   // -128 x the INT2-path fragment values, per group
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        uint32_t lo = 0, hi = 0;   // channels (16ks+2t, +1) and (16ks+2t+8, +9)
        if (g < G) {
            lo = qw[(16 * ks + 2 * t) / 2];
            hi = qw[(16 * ks + 2 * t + 8) / 2];
        }
        const float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&lo));
        const float2 c = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&hi));
        // INT2 path: channels 2t, 2t+8 meet 128 + code; channels 2t+1, 2t+9
        // meet 128 + 4 code and are stored divided by 4 (exact in bf16)
        const uint32_t x0 = (lo & 0xffffu) | (hi << 16);
        const uint32_t x1 = pack2(a.y * 0.25f, c.y * 0.25f);
        if (warp == 0) {
            s_qf[ks * 32 + lane] = make_uint2(lo, hi);
            s_qf[(8 + ks) * 32 + lane] = make_uint2(x0, x1);
        }
        const float2 y1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x1));
        qsum[ks >> 1] += (a.x + a.y) + (c.x + c.y);
        qbias[ks >> 1] -= 128.f * ((a.x + c.x) + (y1.x + y1.y));
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kGroups; ++i) {
        qsum[i] += __shfl_xor_sync(0xffffffffu, qsum[i], 1);
        qsum[i] += __shfl_xor_sync(0xffffffffu, qsum[i], 2);
        qbias[i] += __shfl_xor_sync(0xffffffffu, qbias[i], 1);
        qbias[i] += __shfl_xor_sync(0xffffffffu, qbias[i], 2);
    }
    const float qk_scale = kLog2e * rsqrtf((float)kHeadDim);

    // ---- per-warp online softmax state (lane: head g for m/l, heads 2t, 2t+1 in O)
    float m_run = -INFINITY, l_part = 0.f, w_part = 0.f;
    int n_part = 0;   // partial window entries left by this warp (at most 2)
    float o[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float minacc[kGroups] = {0.f, 0.f, 0.f, 0.f};
    float2 *wstat = S.wstat + ((int64_t)b * Hq + kvh * G) * D.Wmax;

    // ldmatrix row addressing (same for K and V tiles): token and 8-channel half of this lane's row
    const int lm_tok = ((lane >> 4) << 3) + (lane & 7);
    const int lm_hi = (lane >> 3) & 1;

    // online-softmax update with 4 logits of head g (masked ones -inf); turns x into P
    // Online softmax, lazily rescaled: lanes keep partial exp-sums over their own
    // tokens (l_part for the whole run, w_part for the window in progress), both
    // relative to the head's running max m_run, which moves (with a rescale of
    // O, the partial sums and the min accumulators) only when a logit passes it
    // by more than 2^8. Turns the 4 logits of head g in x (masked ones -inf)
    // into P.
    auto softmax4 = [&](float (&x)[4]) {
        const float lmx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
        if (__any_sync(0xffffffffu, lmx > m_run + kLazy)) {
            float hmx = fmaxf(lmx, __shfl_xor_sync(0xffffffffu, lmx, 1));
            hmx = fmaxf(hmx, __shfl_xor_sync(0xffffffffu, hmx, 2));
            const float m_new = fmaxf(m_run, hmx);
            const float alpha = ex2(m_run - m_new);
            m_run = m_new;
            l_part *= alpha;
            w_part *= alpha;
#pragma unroll
            for (int i = 0; i < kGroups; ++i) minacc[i] *= alpha;
            // O columns are heads 2t, 2t+1, whose alphas live in lanes 8t and 8t+4
            const float a_lo = __shfl_sync(0xffffffffu, alpha, 8 * t);
            const float a_hi = __shfl_sync(0xffffffffu, alpha, 8 * t + 4);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                o[i][0] *= a_lo;
                o[i][1] *= a_hi;
                o[i][2] *= a_lo;
                o[i][3] *= a_hi;
            }
        }
        float es = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float e = ex2(x[i] - m_run);
            es += e;
            x[i] = (g < G) ? e : 0.f;
        }
        l_part += es;
        w_part += es;
    };

    while (consumed < issued) {
        const int st = consumed % kStages;
        const bool ok = mbar_wait(smem_u32(&bars[warp][st]), (uint32_t)((consumed / kStages) & 1));
        if (__any_sync(0xffffffffu, !ok)) {
            if (lane == 0) {
                set_status(C, QEVICT_ERR_TIMEOUT, layer, b, consumed);
                for (int r = consumed + 1; r < issued; ++r)
                    (void)mbar_wait(smem_u32(&bars[warp][r % kStages]), (uint32_t)((r / kStages) & 1));
            }
            break;
        }
        __syncwarp();
        const int nb = st_n[warp][st];
        const bool is_fp = st_fp[warp][st] != 0;
        for (int ib = 0; ib < nb; ++ib) {
        const int wi = st_wi[warp][st][ib], ntu = st_nt[warp][st][ib];
        const int emit = st_emit[warp][st][ib];
        const int P = (kWide && !is_fp) ? st_p[warp][st] : 1;
        const uint32_t base = ring_s + st * kStage + ib * (kWide ? (uint32_t)qtile_bytes(P) : (uint32_t)kQUnit);
        if (is_fp) {
            // ---------------- full-precision unit
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int chunk = 2 * (ks & 3) + lm_hi;
                const uint32_t addr = base + (ks >> 2) * 2048 + lm_tok * 128 + ((chunk ^ (lm_tok & 7)) << 4);
                uint32_t b00, b01, b10, b11;
                ldsm_x4(addr, b00, b01, b10, b11);
                const uint2 af = s_qf[ks * 32 + lane];
                mma(s0, af.x, 0u, af.y, 0u, b00, b01);
                mma(s1, af.x, 0u, af.y, 0u, b10, b11);
            }
            float x[4] = {s0[0] * qk_scale, s0[1] * qk_scale, s1[0] * qk_scale, s1[1] * qk_scale};
            if (ntu < 16) {
                // rows past the open window's last token hold stale slot memory: P is 0
                // there, but 0 * NaN would still poison the P.V product, so zero them
                for (int c = lane; c < (16 - ntu) * 16; c += 32) {
                    const int row = ntu + (c >> 4), half = (c >> 3) & 1, ch = c & 7;
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(base + 4096 + half * 2048 +
                                                                                  row * 128 + ch * 16),
                                 "r"(0u)
                                 : "memory");
                }
                __syncwarp();
                if (2 * t >= ntu) x[0] = -INFINITY;
                if (2 * t + 1 >= ntu) x[1] = -INFINITY;
                if (8 + 2 * t >= ntu) x[2] = -INFINITY;
                if (9 + 2 * t >= ntu) x[3] = -INFINITY;
            }
            softmax4(x);
            uint32_t b0h, b0l, b1h, b1l;
            split2(x[0], x[1], b0h, b0l);
            split2(x[2], x[3], b1h, b1l);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const int chunk = 2 * (mt & 3) + lm_hi;
                const uint32_t addr = base + 4096 + (mt >> 2) * 2048 + lm_tok * 128 + ((chunk ^ (lm_tok & 7)) << 4);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(addr, a0, a1, a2, a3);
                mma(o[mt], a0, a1, a2, a3, b0h, b1h);
                mma(o[mt], a0, a1, a2, a3, b0l, b1l);
            }
        } else if (kWide && P == 2) {
            // ---------------- INT4 unit: the two code planes are joined in registers
            // into 4-bit codes (exact in bf16 as 128 + c and 128 + 4 c), then the
            // INT2 unit's arithmetic runs once: same query fragments, same offset
            // correction, 4-bit codes in place of 2-bit ones.
            const uint32_t kc = base, km = base + qtile_kmeta(2), vc = base + qtile_vcodes(2),
                           vm = base + qtile_vmeta(2);
            const int tA = (g & 1) ? g + 7 : g;
            const int tB = (g & 1) ? g + 8 : g + 1;
            uint4 kmeta[4];
            kmeta[0] = lds128(km + (2 * t) * 16);
            kmeta[1] = lds128(km + (2 * t + 8) * 16);
            kmeta[2] = lds128(km + (2 * t + 1) * 16);
            kmeta[3] = lds128(km + (2 * t + 9) * 16);
            float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int grp = 0; grp < kGroups; ++grp) {
                const uint32_t kp = kc + (grp >= 2 ? 16 : 0);
                const uint4 kA0 = lds128(kp + tA * 32), kB0 = lds128(kp + tB * 32);
                const uint4 kA1 = lds128(kp + 512 + tA * 32), kB1 = lds128(kp + 512 + tB * 32);
                float c0[4], c1[4];
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const int ks = 2 * grp + kk;
                    const uint32_t xa0 = pick(kA0, ks & 3) >> (4 * t), xa1 = pick(kA1, ks & 3) >> (4 * t);
                    const uint32_t xb0 = pick(kB0, ks & 3) >> (4 * t), xb1 = pick(kB1, ks & 3) >> (4 * t);
                    const uint2 aq = s_qf[(8 + ks) * 32 + lane];
                    if (kk == 0) {   // start from minus the offsets' share (rows g; rows g + 8 are padding)
                        mma_c(c0, aq.x, 0u, aq.y, 0u, kcodes4_lo(xa0, xa1), kcodes4_hi(xa0, xa1), qbias[grp], 0.f);
                        mma_c(c1, aq.x, 0u, aq.y, 0u, kcodes4_lo(xb0, xb1), kcodes4_hi(xb0, xb1), qbias[grp], 0.f);
                    } else {
                        mma(c0, aq.x, 0u, aq.y, 0u, kcodes4_lo(xa0, xa1), kcodes4_hi(xa0, xa1));
                        mma(c1, aq.x, 0u, aq.y, 0u, kcodes4_lo(xb0, xb1), kcodes4_hi(xb0, xb1));
                    }
                }
                const float acc[4] = {c0[0], c0[1], c1[0], c1[1]};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 sm = h2f(pick(kmeta[i], grp));   // .x scale, .y min
                    x[i] = fmaf(sm.x, acc[i], fmaf(sm.y, qsum[grp], x[i]));
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i] *= qk_scale;
            softmax4(x);
            const int vtok[4] = {2 * t, 2 * t + 8, 2 * t + 1, 2 * t + 9};
#pragma unroll
            for (int grp = 0; grp < kGroups; ++grp) {
                const uint4 vv0 = lds128(vc + g * 64 + grp * 16), vv1 = lds128(vc + 512 + g * 64 + grp * 16);
                uint32_t vmg[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) vmg[i] = lds32(vm + vtok[i] * 16 + grp * 4);
                float val[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 sm = h2f(vmg[i]);
                    val[i] = x[i] * sm.x;
                    minacc[grp] = fmaf(x[i], sm.y, minacc[grp]);
                }
                uint32_t b0h, b0l, b1h, b1l;
                split2(val[0], val[1], b0h, b0l);
                split2(val[2], val[3], b1h, b1l);
#pragma unroll
                for (int mm = 0; mm < 2; ++mm) {
                    const int mt = 2 * grp + mm;
                    const uint32_t x0 = pick(vv0, 2 * mm) >> (4 * t), x1 = pick(vv0, 2 * mm + 1) >> (4 * t);
                    const uint32_t y0 = pick(vv1, 2 * mm) >> (4 * t), y1 = pick(vv1, 2 * mm + 1) >> (4 * t);
                    const uint32_t a0 = codes4(x0, y0), a1 = codes4(x1, y1), a2 = codes4(x0 >> 2, y0 >> 2),
                                   a3 = codes4(x1 >> 2, y1 >> 2);
                    mma(o[mt], a0, a1, a2, a3, b0h, b1h);
                    mma(o[mt], a0, a1, a2, a3, b0l, b1l);
                }
            }
        } else if (kWide && P > 1) {
            // ---------------- INT8 unit: four 2-bit planes, code = c0 + 4 c1 + 16 (c2 + 4 c3).
            // The planes are joined in pairs into two 4-bit nibbles (exact in bf16), and each
            // nibble goes through the INT2 arithmetic with exact codes (no offset), the high
            // one weighted by 16 on the query (K) and on P.scale (V): exact scalings.
            const uint32_t kc = base, km = base + qtile_kmeta(4), vc = base + qtile_vcodes(4),
                           vm = base + qtile_vmeta(4);
            const int tA = (g & 1) ? g + 7 : g;
            const int tB = (g & 1) ? g + 8 : g + 1;
            uint4 kmeta[4];
            kmeta[0] = lds128(km + (2 * t) * 16);
            kmeta[1] = lds128(km + (2 * t + 8) * 16);
            kmeta[2] = lds128(km + (2 * t + 1) * 16);
            kmeta[3] = lds128(km + (2 * t + 9) * 16);
            float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int grp = 0; grp < kGroups; ++grp) {
                float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
                for (int pp = 0; pp < 2; ++pp) {
                    const uint32_t kp = kc + 1024 * pp + (grp >= 2 ? 16 : 0);   // planes 2 pp, 2 pp + 1
                    const uint4 kA0 = lds128(kp + tA * 32), kB0 = lds128(kp + tB * 32);
                    const uint4 kA1 = lds128(kp + 512 + tA * 32), kB1 = lds128(kp + 512 + tB * 32);
                    const __nv_bfloat162 w4 = __float2bfloat162_rn(pp ? 16.f : 1.f);
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const int ks = 2 * grp + kk;
                        const uint32_t xa0 = pick(kA0, ks & 3) >> (4 * t), xa1 = pick(kA1, ks & 3) >> (4 * t);
                        const uint32_t xb0 = pick(kB0, ks & 3) >> (4 * t), xb1 = pick(kB1, ks & 3) >> (4 * t);
                        const uint2 nq = s_qf[ks * 32 + lane];   // natural (q[2t], q[2t+1]), (q[2t+8], q[2t+9])
                        uint32_t a0 = __byte_perm(nq.x, nq.y, 0x5410), a2 = __byte_perm(nq.x, nq.y, 0x7632);
                        __nv_bfloat162 v0 = __hmul2(*reinterpret_cast<__nv_bfloat162 *>(&a0), w4);
                        __nv_bfloat162 v2 = __hmul2(*reinterpret_cast<__nv_bfloat162 *>(&a2), w4);
                        a0 = *reinterpret_cast<uint32_t *>(&v0);
                        a2 = *reinterpret_cast<uint32_t *>(&v2);
                        mma(c0, a0, 0u, a2, 0u, codes4(xa0, xa1), codes4(xa0 >> 2, xa1 >> 2));
                        mma(c1, a0, 0u, a2, 0u, codes4(xb0, xb1), codes4(xb0 >> 2, xb1 >> 2));
                    }
                }
                const float acc[4] = {c0[0], c0[1], c1[0], c1[1]};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 sm = h2f(pick(kmeta[i], grp));   // .x scale, .y min
                    x[i] = fmaf(sm.x, acc[i], fmaf(sm.y, qsum[grp], x[i]));
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i] *= qk_scale;
            softmax4(x);
            const int vtok[4] = {2 * t, 2 * t + 8, 2 * t + 1, 2 * t + 9};
#pragma unroll
            for (int grp = 0; grp < kGroups; ++grp) {
                uint32_t vmg[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) vmg[i] = lds32(vm + vtok[i] * 16 + grp * 4);
                float val[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 sm = h2f(vmg[i]);
                    val[i] = x[i] * sm.x;
                    minacc[grp] = fmaf(x[i], sm.y, minacc[grp]);
                }
                uint32_t b0h, b0l, b1h, b1l;
                split2(val[0], val[1], b0h, b0l);
                split2(val[2], val[3], b1h, b1l);
#pragma unroll 1
                for (int pp = 0; pp < 2; ++pp) {
                    const uint4 vv0 = lds128(vc + 1024 * pp + g * 64 + grp * 16);
                    const uint4 vv1 = lds128(vc + 1024 * pp + 512 + g * 64 + grp * 16);
                    const __nv_bfloat162 w4 = __float2bfloat162_rn(pp ? 16.f : 1.f);
                    uint32_t sc[4] = {b0h, b1h, b0l, b1l};
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        __nv_bfloat162 v = __hmul2(*reinterpret_cast<__nv_bfloat162 *>(&sc[r]), w4);
                        sc[r] = *reinterpret_cast<uint32_t *>(&v);
                    }
#pragma unroll
                    for (int mm = 0; mm < 2; ++mm) {
                        const int mt = 2 * grp + mm;
                        const uint32_t x0 = pick(vv0, 2 * mm) >> (4 * t), x1 = pick(vv0, 2 * mm + 1) >> (4 * t);
                        const uint32_t y0 = pick(vv1, 2 * mm) >> (4 * t), y1 = pick(vv1, 2 * mm + 1) >> (4 * t);
                        const uint32_t a0 = codes4(x0, y0), a1 = codes4(x1, y1), a2 = codes4(x0 >> 2, y0 >> 2),
                                       a3 = codes4(x1 >> 2, y1 >> 2);
                        mma(o[mt], a0, a1, a2, a3, sc[0], sc[1]);
                        mma(o[mt], a0, a1, a2, a3, sc[2], sc[3]);
                    }
                }
            }
        } else {
            // ---------------- INT2 unit
            const uint32_t kc = base, km = base + 512, vc = base + 768, vm = base + 1280;
            // QK: column g of N tile 0 is token tA, of tile 1 token tB
            const int tA = (g & 1) ? g + 7 : g;
            const int tB = (g & 1) ? g + 8 : g + 1;
            const uint4 kA0 = lds128(kc + tA * 32), kA1 = lds128(kc + tA * 32 + 16);
            const uint4 kB0 = lds128(kc + tB * 32), kB1 = lds128(kc + tB * 32 + 16);
            // this lane's logit / probability tokens: 2t, 2t+8 (tile 0), 2t+1, 2t+9 (tile 1)
            uint4 kmeta[4];
            kmeta[0] = lds128(km + (2 * t) * 16);
            kmeta[1] = lds128(km + (2 * t + 8) * 16);
            kmeta[2] = lds128(km + (2 * t + 1) * 16);
            kmeta[3] = lds128(km + (2 * t + 9) * 16);
            float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int grp = 0; grp < kGroups; ++grp) {
                float c0[4], c1[4];
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const int ks = 2 * grp + kk;
                    const uint32_t xa = pick(ks < 4 ? kA0 : kA1, ks & 3) >> (4 * t);
                    const uint32_t xb = pick(ks < 4 ? kB0 : kB1, ks & 3) >> (4 * t);
                    const uint2 aq = s_qf[(8 + ks) * 32 + lane];
                    if (kk == 0) {   // start from minus the offsets' share (rows g; rows g + 8 are padding)
                        mma_c(c0, aq.x, 0u, aq.y, 0u, kcodes_lo(xa), kcodes_hi(xa), qbias[grp], 0.f);
                        mma_c(c1, aq.x, 0u, aq.y, 0u, kcodes_lo(xb), kcodes_hi(xb), qbias[grp], 0.f);
                    } else {
                        mma(c0, aq.x, 0u, aq.y, 0u, kcodes_lo(xa), kcodes_hi(xa));
                        mma(c1, aq.x, 0u, aq.y, 0u, kcodes_lo(xb), kcodes_hi(xb));
                    }
                }
                const float acc[4] = {c0[0], c0[1], c1[0], c1[1]};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 sm = h2f(pick(kmeta[i], grp));   // .x scale, .y min
                    x[i] = fmaf(sm.x, acc[i], fmaf(sm.y, qsum[grp], x[i]));
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i] *= qk_scale;
            softmax4(x);
            // each group's V codes and meta are loaded where they are used,
            // which keeps fewer registers live across the unit
            const int vtok[4] = {2 * t, 2 * t + 8, 2 * t + 1, 2 * t + 9};
#pragma unroll
            for (int grp = 0; grp < kGroups; ++grp) {
                const uint4 vv = lds128(vc + g * 64 + grp * 16);
                uint32_t vmg[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) vmg[i] = lds32(vm + vtok[i] * 16 + grp * 4);
                float val[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 sm = h2f(vmg[i]);
                    val[i] = x[i] * sm.x;
                    minacc[grp] = fmaf(x[i], sm.y, minacc[grp]);
                }
                uint32_t b0h, b0l, b1h, b1l;
                split2(val[0], val[1], b0h, b0l);
                split2(val[2], val[3], b1h, b1l);
                // words of this lane's channels in vv: mt = 2 grp, 2 grp + 1; h = 0 (channel g), 1 (g + 8)
#pragma unroll
                for (int mm = 0; mm < 2; ++mm) {
                    const int mt = 2 * grp + mm;
                    const uint32_t x0 = pick(vv, 2 * mm) >> (4 * t), x1 = pick(vv, 2 * mm + 1) >> (4 * t);
                    const uint32_t a0 = codes2(x0), a1 = codes2(x1), a2 = codes2(x0 >> 2), a3 = codes2(x1 >> 2);
                    mma(o[mt], a0, a1, a2, a3, b0h, b1h);
                    mma(o[mt], a0, a1, a2, a3, b0l, b1l);
                }
            }
        }
        if (emit) {   // (reference max, exp-sum over the window's tokens seen here) for head g
            float ws = w_part + __shfl_xor_sync(0xffffffffu, w_part, 1);
            ws += __shfl_xor_sync(0xffffffffu, ws, 2);
            if (emit == 1) {
                if (t == 0 && g < G) wstat[(int64_t)g * D.Wmax + wi] = make_float2(m_run, ws);
            } else {
                if (t == 0 && g < G) pt_st[warp][n_part][g] = make_float2(m_run, ws);
                if (lane == 0) pt_win[warp][n_part] = wi;
                ++n_part;
            }
            w_part = 0.f;
        }
        }
        __syncwarp();
        ++consumed;
        try_issue();
    }
    __syncthreads();
    // ---- merge the warps (the rings are free now); rows padded by 4 floats
    // so that the fragment stores hit 32 different banks
    constexpr int kOwStride = kHeadDim + 4;
    float *Ow = reinterpret_cast<float *>(smem);                 // [warp][8 heads][kOwStride]
    float *mw_s = Ow + kWarps * 8 * kOwStride;                   // [warp][8]
    float *lw_s = mw_s + kWarps * 8;
    float *minw = lw_s + kWarps * 8;                             // [warp][8][4]
    {
        float *ob = Ow + warp * 8 * kOwStride;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            ob[(2 * t) * kOwStride + 16 * mt + g] = o[mt][0];
            ob[(2 * t + 1) * kOwStride + 16 * mt + g] = o[mt][1];
            ob[(2 * t) * kOwStride + 16 * mt + g + 8] = o[mt][2];
            ob[(2 * t + 1) * kOwStride + 16 * mt + g + 8] = o[mt][3];
        }
    }
#pragma unroll
    for (int i = 0; i < kGroups; ++i) {
        minacc[i] += __shfl_xor_sync(0xffffffffu, minacc[i], 1);
        minacc[i] += __shfl_xor_sync(0xffffffffu, minacc[i], 2);
    }
    l_part += __shfl_xor_sync(0xffffffffu, l_part, 1);
    l_part += __shfl_xor_sync(0xffffffffu, l_part, 2);
    if (t == 0) {
        mw_s[warp * 8 + g] = m_run;
        lw_s[warp * 8 + g] = l_part;
#pragma unroll
        for (int i = 0; i < kGroups; ++i) minw[(warp * 8 + g) * 4 + i] = minacc[i];
    }
    // per-head merge results and the new token, in the free rings
    float *hM = reinterpret_cast<float *>(smem + kHeadOff);                    // [8] max over the splits
    float *hIL = hM + 8;                                                       // [8] 1 / exp-sum
    float *hNew = hIL + 8;                                                     // [8] new token's logit
    float *hFN = hNew + 8;                                                     // [8] new token's weight
    float *Frk = hFN + 8;                                                      // [kMaxSplits][8] weight of each split
    float *sVn = Frk + kMaxSplits * 8;                                         // [128] new token's V row
    const bool has_new = knew != nullptr;
    const __nv_bfloat16 *kn = has_new ? knew + ((int64_t)b * Hkv + kvh) * kHeadDim : nullptr;
    const __nv_bfloat16 *vn = has_new ? vnew + ((int64_t)b * Hkv + kvh) * kHeadDim : nullptr;
    const int64_t Lnew = has_new ? length + 1 : length;
    const int n_out = (int)((Lnew + w - 1) / w);
    const int wnew = (int)(length / w);
    const bool opens = has_new && (length % w == 0);
    // the new token's inputs, requested now and used after the splits meet
    uint2 nq_raw = make_uint2(0u, 0u), nk_raw = make_uint2(0u, 0u);
    __nv_bfloat16 nv_raw = __float2bfloat16(0.f);
    if (has_new) {
        if (warp < G) {
            nq_raw = reinterpret_cast<const uint2 *>(q + ((int64_t)b * Hq + kvh * G + warp) * kHeadDim)[lane];
            nk_raw = reinterpret_cast<const uint2 *>(kn)[lane];
        }
        if (tid < kHeadDim) nv_raw = vn[tid];
    }
    // Every value this split hands to the others leaves as a 64-bit word whose
    // high half is this launch's tag, so a reader tells a current value from a
    // stale one by itself and no fence is needed.
    const uint32_t tag = s_gen + 1u;
    __syncthreads();
    // ---- this split's partial output [G][128] (unnormalised, relative to its
    // own max), one thread per (head, channel); the channel-0 thread of each
    // head also publishes the head's (max, exp-sum) record
    {
        unsigned long long *pacc = S.part + ((int64_t)bk * splits + split) * G * kHeadDim;
        for (int i = tid; i < G * kHeadDim; i += kThreads) {
            const int hh = i / kHeadDim, c = i % kHeadDim;
            float M = -INFINITY;
#pragma unroll
            for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, mw_s[ww * 8 + hh]);
            float acc = 0.f, l = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int ww = 0; ww < kWarps; ++ww) {
                    const float f = ex2(mw_s[ww * 8 + hh] - M);
                    acc = fmaf(f, Ow[(ww * 8 + hh) * kOwStride + c] + minw[(ww * 8 + hh) * 4 + c / kGroup], acc);
                    l = fmaf(f, lw_s[ww * 8 + hh], l);
                }
            }
            const unsigned long long word = ((unsigned long long)tag << 32) | __float_as_uint(acc);
            asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(pacc + i), "l"(word) : "memory");
            if (c == 0) {
                unsigned long long *r = S.rec + ((int64_t)bk * kMaxSplits + split) * kMaxG * 2 + hh * 2;
                const unsigned long long m64 = ((unsigned long long)tag << 32) | __float_as_uint(M);
                const unsigned long long l64 = ((unsigned long long)tag << 32) | __float_as_uint(l);
                asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(r), "l"(m64), "l"(l64) : "memory");
            }
        }
    }
    float *sp = D.score_part + ((int64_t)b * Hkv + kvh) * D.Wmax;
    const int z0 = (int)((int64_t)split * n_out / splits), z1 = (int)((int64_t)(split + 1) * n_out / splits);
    // masses are computed from the top warps down (mt), beside the output
    // work of the low warps
    const int mt = kTailThreads - 1 - tid;
    const uint8_t ztier = (mt >= 0 && z0 + mt < z1) ? D.tier[wb + z0 + mt] : (uint8_t)QEVICT_TIER_E;
    if (warp == kWarps - 1) {
        // this KV head's K and V rows of the new token (split 0), into the
        // slot that receives it: read before this CTA arrives below (the
        // sequence's last CTA moves CTR_NEXT only after every CTA arrived)
        const int slot_new = (!has_new || split != 0) ? -1
                             : opens ? *(volatile const int32_t *)&ctr[CTR_NEXT]
                                     : *(volatile const int32_t *)&D.fp_slot[wb + wnew];
        if (slot_new >= 0) {
            const int row = (int)(length % w);
            const int kv = lane >> 4, c = lane & 15;
            const __nv_bfloat16 *src = kv ? vn : kn;
            __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(D.fp_pool + (int64_t)slot_new * D.fp_slot_bytes) +
                                 fp_off(kvh, kv, w, row, 8 * c);
            *reinterpret_cast<uint4 *>(dst) = reinterpret_cast<const uint4 *>(src)[c];
        }
        if (lane == 0) {
            // Two arrival counts, requested together. Per (sequence, KV head):
            // the last split moves the record generation on for the next
            // launch. Per sequence (fused append only): every CTA of the
            // sequence has read its tables once all have arrived, so the last
            // one moves them forward (tables written only by earlier launches).
            uint32_t *cnt = S.bar + 2 * bk, *gen = cnt + 1;
            const uint32_t prev = atomicAdd(cnt, 1u);
            const unsigned prev_b = has_new ? atomicAdd(&S.arrive_b[b], 1u) : 0u;
            if (prev == (uint32_t)(splits - 1)) {
                *(volatile uint32_t *)cnt = 0u;
                *(volatile uint32_t *)gen = tag;
            }
            if (has_new && prev_b == (unsigned)(Hkv * splits - 1)) {
                int32_t *c = D.ctr + b * kCtrN;
                if (opens) {
                    const int slotn = c[CTR_NEXT];
                    if (slotn < 0) {
                        set_status(C, QEVICT_ERR_CAPACITY, layer, b, wnew);
                    } else {
                        D.tier[wb + wnew] = QEVICT_TIER_FP;
                        D.fp_slot[wb + wnew] = slotn;
                        D.lg_slot[wb + wnew] = -1;
                        D.lwrites[wb + wnew] = 0;
                        const int n = c[CTR_NFP];
                        D.fp_list[b * D.CF + n] = make_int2(wnew, slotn);
                        c[CTR_NFP] = n + 1;
                        const int top = c[CTR_FP_TOP];
                        if (top > 0) {
                            c[CTR_NEXT] = D.fp_free[b * D.CF + top - 1];
                            c[CTR_FP_TOP] = top - 1;
                        } else {
                            c[CTR_NEXT] = -1;
                        }
                    }
                }
                c[CTR_LEN] = (int)Lnew;
                S.arrive_b[b] = 0u;
            }
        }
        return;
    }
    if (warp >= G) {
        // windows cut between warps: entry e = 2 warp + slot; the entries of
        // one window are consecutive among the used ones. One thread per
        // (entry, head) starts at each window's first entry and merges the
        // rest. Done by the warps that do not poll, while the splits meet.
        const int nmw = (kWarps - 1 - G) * 32;
        for (int sl = tid - G * 32; sl < 2 * kWarps * G; sl += nmw) {
            const int e = sl / G, hh = sl % G;
            const int wn = pt_win[e >> 1][e & 1];
            if (wn < 0) continue;
            int pe = e - 1;
            while (pe >= 0 && pt_win[pe >> 1][pe & 1] < 0) --pe;
            if (pe >= 0 && pt_win[pe >> 1][pe & 1] == wn) continue;
            float2 acc = pt_st[e >> 1][e & 1][hh];
            for (int ne = e + 1; ne < 2 * kWarps; ++ne) {
                const int wv = pt_win[ne >> 1][ne & 1];
                if (wv < 0) continue;
                if (wv != wn) break;
                acc = stat_merge(acc, pt_st[ne >> 1][ne & 1][hh]);
            }
            wstat[(int64_t)hh * D.Wmax + wn] = acc;
        }
        asm volatile("bar.sync 2, %0;" ::"r"(nmw) : "memory");
    }
    // statistics of the first window of each mass thread of those warps (all
    // in global memory now) and its old score, fetched while the splits meet
    const bool pre = warp >= G && mt < nwin;
    int pwi = -1;
    float pold = 0.f;
    float2 pst[G];
    if (pre) {
        pwi = ent(mt).x;
#pragma unroll
        for (int hh = 0; hh < G; ++hh) pst[hh] = wstat[(int64_t)hh * D.Wmax + pwi];
        pold = accumulate ? sp[pwi] : 0.f;
    }
    // ---- output gather: this split's slice of the [G][32] float4 outputs,
    // one (output, split) item per thread of the warps that do not poll. Each
    // waits until the four tagged words of its item are current and keeps the
    // raw values; they are weighted and summed once the splits have met.
    const int n4 = G * (kHeadDim / 4);
    const int o0 = split * n4 / splits, o1 = (split + 1) * n4 / splits;
    const int nwork = (o1 - o0) * splits;
    float4 *red = reinterpret_cast<float4 *>(smem + kRedOff);   // [outputs of the slice][splits]
    if (warp >= G) {
        const unsigned long long *pw = S.part + (int64_t)bk * splits * G * kHeadDim;
        bool ok = true;
        for (int t = tid - G * 32; t < nwork; t += (kWarps - 1 - G) * 32) {
            const int oi = o0 + t / splits, r = t % splits;
            const int hh = oi / (kHeadDim / 4), c4 = oi % (kHeadDim / 4);
            const unsigned long long *a4 = pw + ((int64_t)r * G + hh) * kHeadDim + 4 * c4;
            unsigned long long u0, u1, u2, u3;
            const long long t0 = clock64();
            while (true) {
                asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(u0), "=l"(u1) : "l"(a4) : "memory");
                asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(u2), "=l"(u3) : "l"(a4 + 2) : "memory");
                if ((uint32_t)(u0 >> 32) == tag && (uint32_t)(u1 >> 32) == tag && (uint32_t)(u2 >> 32) == tag &&
                    (uint32_t)(u3 >> 32) == tag)
                    break;
                if (clock64() - t0 > kWaitCycles) {
                    ok = false;
                    break;
                }
                __nanosleep(32);
            }
            red[t] = ok ? make_float4(__uint_as_float((uint32_t)u0), __uint_as_float((uint32_t)u1),
                                      __uint_as_float((uint32_t)u2), __uint_as_float((uint32_t)u3))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (!ok) set_status(C, QEVICT_ERR_TIMEOUT, layer, b, -4);
    }
    // max and exp-sum over the splits: warp hh polls head hh's records (lane = split)
    if (warp < G) {
        const int hh = warp;
        float nl = -INFINITY;   // the new token's logit
        if (has_new) {
            const float2 q0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&nq_raw.x));
            const float2 q1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&nq_raw.y));
            const float2 k0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&nk_raw.x));
            const float2 k1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&nk_raw.y));
            float d = fmaf(q0.x, k0.x, fmaf(q0.y, k0.y, fmaf(q1.x, k1.x, q1.y * k1.y)));
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o2);
            nl = d * qk_scale;
        }
        float2 v = make_float2(-INFINITY, 0.f);
        bool ok = true;
        if (lane < splits) {
            const unsigned long long *r = S.rec + ((int64_t)bk * kMaxSplits + lane) * kMaxG * 2 + hh * 2;
            unsigned long long m64, l64;
            const long long t0 = clock64();
            while (true) {
                asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(m64), "=l"(l64) : "l"(r) : "memory");
                if ((uint32_t)(m64 >> 32) == tag && (uint32_t)(l64 >> 32) == tag) break;
                if (clock64() - t0 > kWaitCycles) {
                    ok = false;
                    break;
                }
                __nanosleep(32);
            }
            v = ok ? make_float2(__uint_as_float((uint32_t)m64), __uint_as_float((uint32_t)l64))
                   : make_float2(-INFINITY, 0.f);
        }
        if (__any_sync(0xffffffffu, !ok) && lane == 0) set_status(C, QEVICT_ERR_TIMEOUT, layer, b, -3);
        float M = v.x;
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
        if (has_new) M = fmaxf(M, nl);
        const float f = (lane < splits && M != -INFINITY && v.x != -INFINITY) ? ex2(v.x - M) : 0.f;
        if (lane < splits) Frk[lane * 8 + hh] = f;
        float l = f * v.y;
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o2);
        if (lane == 0) {
            const float fn = has_new ? ex2(nl - M) : 0.f;
            l += fn;
            hM[hh] = M;
            hIL[hh] = l > 0.f ? 1.f / l : 0.f;
            hFN[hh] = fn;
            hNew[hh] = nl;
        }
    }
    if (has_new && tid < kHeadDim) sVn[tid] = __bfloat162float(nv_raw);
    tail_sync();
    // output: weight the gathered partials by their splits' factors and sum
    for (int t = tid; t < o1 - o0; t += kTailThreads) {
        const int oi = o0 + t;
        const int hh = oi / (kHeadDim / 4), c4 = oi % (kHeadDim / 4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (has_new) {
            const float fn = hFN[hh];
            acc = make_float4(fn * sVn[4 * c4], fn * sVn[4 * c4 + 1], fn * sVn[4 * c4 + 2], fn * sVn[4 * c4 + 3]);
        }
        for (int r = 0; r < splits; ++r) {
            const float f = Frk[r * 8 + hh];
            const float4 v = red[t * splits + r];
            acc.x = fmaf(f, v.x, acc.x);
            acc.y = fmaf(f, v.y, acc.y);
            acc.z = fmaf(f, v.z, acc.z);
            acc.w = fmaf(f, v.w, acc.w);
        }
        const float il = hIL[hh];
        reinterpret_cast<float4 *>(out + ((int64_t)b * Hq + kvh * G + hh) * kHeadDim)[c4] =
            make_float4(acc.x * il, acc.y * il, acc.z * il, acc.w * il);
    }

    // ---- masses and cumulative scores of this split's windows
    const float inv_hq = 1.f / (float)Hq;
    for (int li = mt; li < nwin; li += kTailThreads) {
        int wi = pwi;
        float old = pold;
        float2 st[G];
        if (li == mt && pre) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) st[hh] = pst[hh];
        } else {
            wi = ent(li).x;
#pragma unroll
            for (int hh = 0; hh < G; ++hh) st[hh] = wstat[(int64_t)hh * D.Wmax + wi];
            old = accumulate ? sp[wi] : 0.f;
        }
        float sum = 0.f;
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            float2 stt = st[hh];
            if (has_new && wi == wnew) stt = stat_merge(stt, make_float2(hNew[hh], 1.f));   // the new token's window
            const float m = (hM[hh] != -INFINITY && stt.y > 0.f) ? stt.y * ex2(stt.x - hM[hh]) * hIL[hh] : 0.f;
            if (mass) mass[((int64_t)b * Hq + kvh * G + hh) * n_out + wi] = m;
            sum += m;
        }
        if (accumulate) sp[wi] = old + sum * inv_hq;
    }
    // windows no split holds: evicted ones (mass 0) and a window this step
    // opens; the window range is sliced over the splits
    for (int wi = z0 + mt; wi < z1; wi += kTailThreads) {
        const bool fresh = opens && wi == wnew;
        if (!fresh && (wi == z0 + mt ? ztier : D.tier[wb + wi]) != QEVICT_TIER_E) continue;
        float sum = 0.f;
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            const float m = (fresh && hM[hh] != -INFINITY) ? ex2(hNew[hh] - hM[hh]) * hIL[hh] : 0.f;
            if (mass) mass[((int64_t)b * Hq + kvh * G + hh) * n_out + wi] = m;
            sum += m;
        }
        if (accumulate && fresh) sp[wi] += sum * inv_hq;
    }
}

constexpr int kDynSmem = kWarps * kRing + kEntTab * 8 + 16 * 32 * 8 + 1024;

// CTAs of decode_kernel<G> that fit on one SM, filled in by prepare_decode.
int g_ctas_per_sm[kMaxG + 1];

template <int G, bool kWide>
cudaError_t prepare_inst(int optin, int *per_sm) {
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, decode_kernel<G, kWide>);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_kernel<G, kWide>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - (int)fa.sharedSizeBytes);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, decode_kernel<G, kWide>, kThreads, kDynSmem);
}
// Both instantiations must fit as many CTAs per SM as the split count assumes.
template <int G>
cudaError_t prepare_one(int optin) {
    int a = 0, w = 0;
    cudaError_t e = prepare_inst<G, false>(optin, &a);
    if (e == cudaSuccess) e = prepare_inst<G, true>(optin, &w);
    g_ctas_per_sm[G] = a < w ? a : w;
    return e;
}

}  // namespace

// Raise the dynamic shared-memory limit of every decode instantiation and
// record how many of its CTAs fit on one SM (called at cache creation,
// outside any stream capture).
cudaError_t prepare_decode() {
    return once_per_device(0, []() {
        int dev = 0, optin = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e == cudaSuccess) e = prepare_one<1>(optin);
        if (e == cudaSuccess) e = prepare_one<2>(optin);
        if (e == cudaSuccess) e = prepare_one<3>(optin);
        if (e == cudaSuccess) e = prepare_one<4>(optin);
        if (e == cudaSuccess) e = prepare_one<5>(optin);
        if (e == cudaSuccess) e = prepare_one<6>(optin);
        if (e == cudaSuccess) e = prepare_one<7>(optin);
        if (e == cudaSuccess) e = prepare_one<8>(optin);
        return e;
    });
}

// Splits per (sequence, KV head): as many as keep the whole grid resident at
// once (the splits of a pair wait for one another), at most kMaxSplits.
int decode_splits(int pairs, int num_sms, int G) {
    const int per_sm = (G >= 1 && G <= kMaxG && g_ctas_per_sm[G] > 0) ? g_ctas_per_sm[G] : 1;
    int s = per_sm * num_sms / (pairs > 0 ? pairs : 1);
    if (s > kMaxSplits) s = kMaxSplits;
    if (s < 1) s = 1;
    return s;
}

cudaError_t launch_decode(const LayerDev &L, const CacheDev &C, const DecodeScratch &S, const CUtensorMap &tmap,
                          int layer, const __nv_bfloat16 *q, const __nv_bfloat16 *knew, const __nv_bfloat16 *vnew,
                          float *out, float *mass, int accumulate, int splits, bool pdl, cudaStream_t s) {
    const bool wide = L.maxP > 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(splits, L.B * L.Hkv);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kDynSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
#define QV_CASE(GG)                                                                                          \
    case GG:                                                                                                 \
        return wide ? cudaLaunchKernelEx(&cfg, decode_kernel<GG, true>, L, C, S, tmap, layer, q, knew, vnew,  \
                                         out, mass, accumulate, splits)                                      \
                    : cudaLaunchKernelEx(&cfg, decode_kernel<GG, false>, L, C, S, tmap, layer, q, knew, vnew, \
                                         out, mass, accumulate, splits);
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
}

}  // namespace qevict
