// Split-K single-token GQA decode attention over the three-tier cache, with
// the per-window softmax mass, the cumulative-score update and (optionally)
// the append of this step's token.
//
// Method: "Technische Samenvatting: QEvict" (gist.science 2608.05326),
// "Methodologie: QEvict" (full-precision and INT2 windows stay visible to
// attention, evicted windows do not) and "Kernmechanismen" (cumulative
// scoring, GQA). "Technische Samenvatting: LogQuant" (gist.science
// 2503.19950), Methodologie 3 and 4: evicted tokens leave the softmax
// normalisation, and cache entries may be visited in any order.
//
// Grid (splits, B * Hkv), one 12-warp CTA per SM and the whole grid resident
// in one wave. A CTA takes a proportional share of one (sequence, KV head)'s
// quantised windows and of its full-precision windows. The work is a list of
// claims: quantised chunks (up to four 16-token tiles of one window, one bulk
// copy; the chunk size shrinks to give about two claims per warp) interleaved
// evenly with full-precision units (16 tokens, K and V in one 4-D TMA tile
// load, 128-byte swizzled). The prologue writes one descriptor per claim into
// shared memory; the warps take claims from a shared-memory counter, each
// into its own ring of two 8 KiB stages, so the work evens out inside the CTA.
// Per 16 tokens a warp computes, on the tensor cores (mma.sync m16n8k16, fp32
// accumulation):
//  - QK with the tokens as the M rows and the query heads as the N columns
//    (for G <= 4 every head fills two columns). INT2 codes become exact bf16
//    operands in registers (128 + c, or 128 + 4c where the query value is
//    stored divided by 4); the offsets' share is the accumulator's start
//    value. Per group of 32 channels the scale multiplies the group's
//    accumulator; the minimum's share, sum over groups of min_g * (sum of q
//    over g), is one fp16 MMA of the minimums against the per-group query
//    sums split into fp16 hi + lo. The result is the real-valued
//    reconstruction min + code * scale up to fp32 rounding.
//  - softmax in the log2 domain with a running max per head that moves only
//    when a logit passes it by more than 2^8.
//  - PV as O^T = V^T P: channels as M, tokens as K, heads as N. P (times the
//    token's V scale for INT2) is split into bf16 hi + lo; for G <= 4 the hi
//    parts fill columns 0-3 and the lo parts columns 4-7 of one MMA (the
//    duplicated QK columns hold the same probabilities), otherwise two MMAs.
//    movmatrix transposes P from the QK result layout into the operand
//    layout. The V minimum's share is a CUDA-core sum per group.
//  The token order inside a quantised tile follows the V code words (pairs
//  of tokens share a 32-bit word), and the same order is used on both sides
//  of each product, which leaves every sum unchanged. After each claim the
//  warp stores the claim's (reference max, exp-sum) per head as a record.
//
// The wide instantiation (decode_kernel<G, true>, caches that allow INT4 and
// INT8 windows, "Technische Samenvatting: RDKV", 2.2 and 2.3) reads a window
// of b bits as b / 2 two-bit code planes: INT4 joins its two planes into 4-bit
// codes in registers and runs the INT2 arithmetic once, INT8 runs it on two
// nibbles, the high one weighted 16. Its claims take as many tiles of a window
// as a stage holds at the window's width, and each chunk runs the arithmetic
// compiled for its plane count. On a layer with K-channel widths each
// 32-channel K group is read at its own width (width 0: skipped).
//
// After the loop the warps merge in shared memory and the CTA publishes its
// partial output and (max, exp-sum) per head as 64-bit words tagged with the
// launch's generation. The splits of a (sequence, KV head) meet on those
// records (bounded polls), then each writes a slice of the merged output, the
// masses of its own windows (from its records; their mean over the Hq heads
// grows the KV head's partial cumulative score) and the zero masses of its
// slice of the evicted windows. With a new token, split 0 writes its K and V
// rows into their slot, and once every CTA of the sequence has published, split
// 0 of KV head 0 opens the new window and moves the length.
//
// With programmatic dependent launch the kernel reads its window lists and
// issues its first copies before it waits for the previous kernel
// (griddepcontrol.wait); it reads the query and the scratch only after.
#include "qevict_internal.cuh"

namespace qevict {

namespace {

constexpr int kWarps = 12;                // warps per decode CTA (one CTA per SM)
constexpr int kThreads = kWarps * 32;
constexpr int kSlots = 2;                 // ring slots per warp
constexpr int kSlot = 8192;               // bytes per slot: a full-precision unit (16 tokens, K and V)
                                          // or up to five quantised tiles
constexpr int kRing = kSlots * kSlot;
constexpr int kQChunk = 5;                // INT2 tiles per stage at most (7.5 KiB)
constexpr int kDescTab = 1024;            // claim descriptors of a split kept in shared memory
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.f;              // log2 headroom before the running max moves
constexpr long long kWaitCycles = kDefaultWaitCycles;   // waits on this CTA's own copies
// ring stage: quantised chunk, full-precision unit, a claim of no tokens
enum { EL_Q = 0, EL_F = 1, EL_SKIP = 3 };

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
// D += A B (bf16 operands, fp32 accumulators)
__device__ __forceinline__ void mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                    uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D = A B + C with C = {c0, c1, c0, c1} (one start value per N column)
__device__ __forceinline__ void mma_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                      uint32_t b1, float c0, float c1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %11, %10, %11};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1));
}
// D = A B with fp16 operands; A's k columns 8..15 and B's k rows 8..15 zero
__device__ __forceinline__ void mma_f16_k8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %6}, {%7, %6}, "
        "{%8, %8, %8, %8};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(0u), "r"(b0), "f"(0.f));
}
// 8x8 b16 transpose across the warp: lane 4r + c holds row r, columns 2c, 2c + 1
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
// shared-memory loads through typed pointers, so that the compiler may schedule them
__device__ __forceinline__ uint32_t ld32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }
__device__ __forceinline__ uint2 ld64(const uint8_t *p) { return *reinterpret_cast<const uint2 *>(p); }
__device__ __forceinline__ uint4 ld128(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }
__device__ __forceinline__ uint32_t pick(const uint4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}
__device__ __forceinline__ uint32_t bsub128(uint32_t r) {   // each bf16 half minus 128 (exact)
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&r);
    v = __hsub2(v, __floats2bfloat162_rn(128.f, 128.f));
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t bmul16(uint32_t r) {    // each bf16 half times 16 (exact)
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&r);
    v = __hmul2(v, __floats2bfloat162_rn(16.f, 16.f));
    return *reinterpret_cast<uint32_t *>(&v);
}
// Code words: bits 1:0 and 17:16 of x (after the lane's shift) are two codes,
// bits 3:2 and 19:18 two more. As bf16 pairs with the offset kept: 128 + c
// and 128 + 4c (exact); without it (minus 128): c and 4c. The offset pattern
// k = 0x43004300 comes in a register, so that each pair is one three-input
// logic op (mask immediate, offset register).
template <uint32_t M>
__device__ __forceinline__ uint32_t and_or(uint32_t x, uint32_t k) {   // (x & M) | k
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "n"(M), "r"(k));
    return d;
}
__device__ __forceinline__ uint32_t off_lo(uint32_t x, uint32_t k) { return and_or<0x00030003u>(x, k); }
__device__ __forceinline__ uint32_t off_hi(uint32_t x, uint32_t k) { return and_or<0x000C000Cu>(x, k); }
// 4-bit codes c = c0 + 4 c1 from two planes (x0: c0, x1: c1 at the same positions)
__device__ __forceinline__ uint32_t off4_lo(uint32_t x0, uint32_t x1, uint32_t k) {
    return and_or<0x00030003u>(x0, and_or<0x000C000Cu>(x1 << 2, k));
}
__device__ __forceinline__ uint32_t off4_hi(uint32_t x0, uint32_t x1, uint32_t k) {
    return and_or<0x000C000Cu>(x0, and_or<0x00300030u>(x1 << 2, k));
}
__device__ __forceinline__ uint32_t pack_rn(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
// bf16 hi = rn(x) and lo = rn(x - hi) of a pair: hi + lo is x within 2^-17 relative
__device__ __forceinline__ void split_pair(float a, float b, uint32_t &hi, uint32_t &lo) {
    hi = pack_rn(a, b);
    lo = pack_rn(a - bf_lo(hi), b - bf_hi(hi));
}
// the hi part on hi lanes (lo_f = 0), the lo part on lo lanes (lo_f = 1), without a branch
__device__ __forceinline__ uint32_t split_sel(float a, float b, float lo_f) {
    const uint32_t hi = pack_rn(a, b);
    return pack_rn(fmaf(-lo_f, bf_lo(hi), a), fmaf(-lo_f, bf_hi(hi), b));
}
__device__ __forceinline__ float2 h2f(uint32_t u) {
    const __half2 h = *reinterpret_cast<const __half2 *>(&u);
    return __half22float2(h);
}
// 2^x (PTX ex2.approx; results below 2^-126 flush to zero)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr int kRecMax = 8;     // records per window: 16-token tiles (w <= 128)

// A code-plane count known at compile time (converts to its int)
template <int P>
struct PlanesC {
    __device__ constexpr operator int() const { return P; }
};

// One split's claims (see decode_kernel): whole quantised windows [qw0, qw0 +
// nqw) and whole full-precision windows [fw0, fw0 + nfw), i.e. units [f0, f0 +
// nfl), of one (sequence, KV head).
struct ClaimPlan {
    int64_t length;
    int n_win, qw0, nqw, fw0, nfw, f0, nfl, tpc, cpw, tailw, nbig, N;
    int kcodes;   // K code bytes of a K-channel tile of this KV head, or -1 (plane tiles)
};

template <bool kWide>
__device__ __forceinline__ ClaimPlan claim_plan(const LayerDev &D, int b, int kvh, int split, int splits, int mu) {
    const int32_t *ctr = D.ctr + b * kCtrN;
    ClaimPlan p;
    p.length = ctr[CTR_LEN];
    p.kcodes = (kWide && ctr[CTR_KCH] != 0) ? ktile_kcodes(D.kgw + ((int64_t)b * D.Hkv + kvh) * kGroups) : -1;
    const int n_fp = ctr[CTR_NFP], n_q = ctr[CTR_NQ];
    p.n_win = (int)((p.length + D.w - 1) / D.w);
    // (window counts are at most 4096 and splits at most 32: 32-bit products suffice)
    p.qw0 = (int)((unsigned)n_q * split / splits);
    p.nqw = (int)((unsigned)n_q * (split + 1) / splits) - p.qw0;
    p.fw0 = (int)((unsigned)n_fp * split / splits);
    p.nfw = (int)((unsigned)n_fp * (split + 1) / splits) - p.fw0;
    p.f0 = p.fw0 * mu;
    p.nfl = p.nfw * mu;
    {
        // tiles per chunk: at most what one stage holds, and about two claims per warp
        const int fit = mu <= kQChunk ? mu : (mu + 1) / 2;
        p.tpc = kWide ? 1 : max(1, min(fit, (p.nqw * mu) / (2 * kWarps)));
    }
    p.cpw = (mu + p.tpc - 1) / p.tpc;                     // chunks per window
    p.tailw = 0;   // (single-tile claims for the last windows: none)
    p.nbig = (p.nqw - p.tailw) * p.cpw;
    p.N = p.nbig + p.tailw * mu + p.nfl;
    return p;
}

// Descriptor of claim c: {kind | n << 2 | log2 P << 7, record slot, z, w}. A
// quantised chunk of n tiles has z = (byte offset of its tiles in the ledger
// pool) / 512 and w = its bytes; a full-precision unit of n tokens has z, w =
// the TMA coordinates of its tile (slot * Hkv + kvh, 16 j).
// Descriptor of the split's full-precision unit fb.
__device__ __forceinline__ int4 fp_desc(const LayerDev &D, const ClaimPlan &p, int b, int kvh, int mu, int fb) {
    const int w = D.w;
    const int gf = p.f0 + fb, e = gf / mu, j = gf - e * mu;
    const int2 en = D.fp_list[b * D.CF + e];
    const int nt = ((en.x == p.n_win - 1) ? (int)(p.length - (int64_t)en.x * w) : w) - 16 * j;
    if (nt <= 0) return make_int4(EL_SKIP, 0, 0, 0);   // past the open window's last token
    return make_int4(EL_F | (min(16, nt) << 2), e * mu + j, en.y * D.Hkv + kvh, 16 * j);
}

template <bool kWide>
__device__ __forceinline__ int4 claim_desc(const LayerDev &D, const ClaimPlan &p, int b, int kvh, int mu, int c) {
    const int w = D.w;
    // a split has at most 2^16 claims and 2^15 full-precision units: the products fit 32 bits
    const int fb = (int)((unsigned)c * p.nfl / p.N);
    if ((int)((unsigned)(c + 1) * p.nfl / p.N) > fb) return fp_desc(D, p, b, kvh, mu, fb);
    const int ci = c - fb;
    int k, u0, n;
    if (ci < p.nbig) {
        k = ci / p.cpw;
        u0 = (ci - k * p.cpw) * p.tpc;
        n = min(p.tpc, mu - u0);
    } else {
        const int c2 = ci - p.nbig;
        k = p.nqw - p.tailw + c2 / mu;
        u0 = c2 - (c2 / mu) * mu;
        n = 1;
    }
    const int e = p.qw0 + k;
    const int2 en = D.q_list[b * D.CQ + e];
    const int lgP = kWide ? (en.y >> kSlotBits) : 0;
    const int slot = kWide ? (en.y & ((1 << kSlotBits) - 1)) : en.y;
    const int P = 1 << lgP;
    if (kWide && p.kcodes >= 0) {   // K-channel tiles sit at the widest tile's stride
        const int64_t off = (int64_t)slot * D.lg_slot_bytes + ((int64_t)kvh * mu + u0) * qtile_bytes(4);
        return make_int4(EL_Q | (n << 2) | (lgP << 7), D.CF * mu + e * mu + u0, (int)(off >> 9),
                         n * ktile_bytes(p.kcodes, P));
    }
    const int64_t off = (int64_t)slot * D.lg_slot_bytes + lg_tile_off(kvh, w, u0, P);
    return make_int4(EL_Q | (n << 2) | (lgP << 7), D.CF * mu + e * mu + u0, (int)(off >> 9), n * qtile_bytes(P));
}

// Wide plane tiles in chunks: a claim takes up to `tpc` tiles of one window,
// at most what one stage holds at the window's width. Quantised claim ci
// belongs to the window k with pref[k] <= ci < pref[k + 1] (pref: exclusive
// prefix of the claims per window), interleaved with the full-precision units
// as in claim_desc over N claims.
__device__ __forceinline__ int wide_tpc(int P, int mu, int target) {
    return min(target, min(mu, kSlot / qtile_bytes(P)));
}
__device__ __forceinline__ int4 chunk_desc(const LayerDev &D, const ClaimPlan &p, int kvh, int mu, int c, int N,
                                           const int *pref, const int *qy, const int2 *fpe, int target) {
    const int fb = (int)((unsigned)c * p.nfl / N);
    if ((int)((unsigned)(c + 1) * p.nfl / N) > fb) {   // full-precision unit fb (its list entry in fpe)
        const int gf = p.f0 + fb, e = gf / mu, j = gf - e * mu;
        const int2 en = fpe[e - p.fw0];
        const int nt = ((en.x == p.n_win - 1) ? (int)(p.length - (int64_t)en.x * D.w) : D.w) - 16 * j;
        if (nt <= 0) return make_int4(EL_SKIP, 0, 0, 0);   // past the open window's last token
        return make_int4(EL_F | (min(16, nt) << 2), e * mu + j, en.y * D.Hkv + kvh, 16 * j);
    }
    const int ci = c - fb;
    int lo = 0, hi = p.nqw - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pref[mid] <= ci)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int e = p.qw0 + lo;
    const int ey = qy[lo];   // the window's list entry .y: log2 planes, slot
    const int lgP = ey >> kSlotBits, slot = ey & ((1 << kSlotBits) - 1), P = 1 << lgP;
    const int tpc = wide_tpc(P, mu, target);
    const int u0 = (ci - pref[lo]) * tpc, n = min(tpc, mu - u0);
    const int64_t off = (int64_t)slot * D.lg_slot_bytes + lg_tile_off(kvh, D.w, u0, P);
    return make_int4(EL_Q | (n << 2) | (lgP << 7), D.CF * mu + e * mu + u0, (int)(off >> 9), n * qtile_bytes(P));
}

// kWide: the cache may hold INT4 / INT8 windows (2 or 4 code planes) or
// K-channel tiles; then the tiles per claim follow each window's width
// (wide_tpc; K-channel tiles one per claim), and each chunk runs the
// arithmetic of its plane count. The instantiation without it is the INT2 /
// full-precision kernel as such.
//
// A split's share of a (sequence, KV head)'s work is a proportional share of
// each list: whole quantised windows [qw0, qw1) and full-precision units
// [f0, f1), so compute-bound and bandwidth-bound work mix evenly over the
// CTAs. Its claim list interleaves the two evenly; a quantised window is
// claimed in chunks of up to four tiles, except the last windows of the
// share, which go one tile at a time so that the warps finish together. The
// prologue writes one descriptor per claim into shared memory.
template <int G, bool kWide>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const LayerDev D, const CacheDev C, const DecodeScratch S, const __grid_constant__ CUtensorMap tmap,
                  int layer, const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *knew,
                  const __nv_bfloat16 *vnew, float *__restrict__ out, float *__restrict__ mass, int accumulate,
                  int splits) {
    constexpr bool kDup = G <= 4;   // every head fills two N columns: hi and lo parts of P share one PV MMA
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 128-byte-swizzled TMA tiles need 1024-byte aligned destinations
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    int4 *s_desc = reinterpret_cast<int4 *>(smem + kWarps * kRing);   // claim descriptors
    // query B fragments per lane: [path (0 natural, 1 INT2 channel order)][k-step][lane] {b0, b1}
    uint2 *s_qf = reinterpret_cast<uint2 *>(smem + kWarps * kRing + kDescTab * 16);
    float2 *s_qb = reinterpret_cast<float2 *>(smem + kWarps * kRing + kDescTab * 16 + 16 * 32 * 8);   // [grp][t]
    __shared__ uint64_t bars[kWarps][kSlots];
    __shared__ int sl_kind[kWarps][kSlots];   // EL_*
    __shared__ int sl_n[kWarps][kSlots];      // tiles of a quantised chunk, tokens of a full-precision unit
    __shared__ int sl_id[kWarps][kSlots];     // record slot of the chunk / unit
    __shared__ int sl_p[kWarps][kSlots];      // code planes of a quantised chunk (kWide)
    __shared__ int s_next;                    // next claim
    __shared__ int s_span[4];                 // this split's quantised and full-precision windows
    __shared__ long long s_len;               // the sequence's length at launch
    __shared__ int s_slot_new;                // slot of the new token's window (split 0, fused append)
    __shared__ uint32_t s_gen;                // split-record generation of this launch
    __shared__ int s_kg[9];                   // K-channel tiles: planes and code offset of each group, code bytes
    __shared__ int s_ws[kWarps];              // per-warp sums of the chunk scan

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int split = blockIdx.x, bk = blockIdx.y;
    const int Hkv = D.Hkv, Hq = D.Hq, w = D.w, mu = w / 16;
    const int b = bk / Hkv, kvh = bk % Hkv;
    float2 *rec = S.rec + (int64_t)bk * S.rec_stride * G;
    const uint32_t ring_s = smem_u32(smem + warp * kRing);

    // ---- claim descriptors, built by all threads at once
    const int N = [&]() {
        const ClaimPlan p = claim_plan<kWide>(D, b, kvh, split, splits, mu);
        int n_claims = p.N;
        bool chunked = false;
        if (kWide && p.kcodes < 0 && p.nqw > 0) {
            // wide plane tiles: several tiles of a window per claim (wide_tpc); the claims per
            // window are prefix-summed in the ring space, which no copy has reached yet, beside
            // the split's list entries (at most 4096 windows: 32 KB), read once here
            int *pref = reinterpret_cast<int *>(smem);
            int *qy = pref + p.nqw;
            int2 *fpe = reinterpret_cast<int2 *>(qy + p.nqw);   // 8-byte aligned: 8 nqw bytes in
            for (int i = tid; i < p.nfw; i += kThreads) fpe[i] = D.fp_list[b * D.CF + p.fw0 + i];
            const int target = max(1, (p.nqw * mu) / (2 * kWarps));
            const int per = (p.nqw + kThreads - 1) / kThreads;
            const int k0 = min(p.nqw, tid * per), k1 = min(p.nqw, k0 + per);
            int cnt = 0;
            for (int k = k0; k < k1; ++k) {
                const int ey = D.q_list[b * D.CQ + p.qw0 + k].y;
                qy[k] = ey;
                const int tpc = wide_tpc(1 << (ey >> kSlotBits), mu, target);
                pref[k] = (mu + tpc - 1) / tpc;
                cnt += pref[k];
            }
            int x = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (lane == 31) s_ws[warp] = x;
            __syncthreads();
            int run = x - cnt, total = 0;
            for (int i = 0; i < kWarps; ++i) {
                run += i < warp ? s_ws[i] : 0;
                total += s_ws[i];
            }
            for (int k = k0; k < k1; ++k) {
                const int cw = pref[k];
                pref[k] = run;
                run += cw;
            }
            __syncthreads();
            if (total + p.nfl <= kDescTab) {
                chunked = true;
                n_claims = total + p.nfl;
                for (int c = tid; c < n_claims; c += kThreads)
                    s_desc[c] = chunk_desc(D, p, kvh, mu, c, n_claims, pref, qy, fpe, target);
            }
        }
        if (!chunked)
            for (int c = tid; c < min(p.N, kDescTab); c += kThreads) s_desc[c] = claim_desc<kWide>(D, p, b, kvh, mu, c);
        if (tid == 0) {
            s_span[0] = p.qw0;
            s_span[1] = p.nqw;
            s_span[2] = p.fw0;
            s_span[3] = p.nfw;
            s_len = p.length;
            s_kg[8] = p.kcodes;
            if (kWide && p.kcodes >= 0) {
                const uint8_t *kw = D.kgw + ((int64_t)b * Hkv + kvh) * kGroups;
                int off = 0;
                for (int gg = 0; gg < kGroups; ++gg) {
                    s_kg[gg] = kgroup_planes(kw[gg]);
                    s_kg[4 + gg] = off;
                    off += 128 * s_kg[gg];
                }
            }
            if (knew != nullptr && split == 0 && p.length < D.max_context) {
                const int64_t wn = p.length / w;
                s_slot_new = (p.length % w == 0) ? D.ctr[b * kCtrN + CTR_NEXT] : D.fp_slot[(int64_t)b * D.Wmax + wn];
            }
        }
        return n_claims;
    }();
    if (lane == 0)
        for (int i = 0; i < kSlots; ++i) mbar_init(smem_u32(&bars[warp][i]), 1);
    if (tid == 0) s_next = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();
    // ---- issue: lane 0 claims and issues, every lane follows the bookkeeping
    const uint64_t l2_stream = evict_first_policy();
    int issued = 0, consumed = 0;
    bool drained = false;                  // no claim left
    auto try_issue = [&]() {
        while (issued - consumed < kSlots) {
            const int sl = issued % kSlots;
            const uint32_t bar = smem_u32(&bars[warp][sl]);
            const uint32_t dst = ring_s + sl * kSlot;
            if (drained) break;
            int c = 0;
            if (lane == 0) c = atomicAdd(&s_next, 1);
            c = __shfl_sync(0xffffffffu, c, 0);
            if (c >= N) {
                drained = true;
                break;
            }
            const int4 d = c < kDescTab ? s_desc[c]
                                        : claim_desc<kWide>(D, claim_plan<kWide>(D, b, kvh, split, splits, mu), b,
                                                            kvh, mu, c);
            const int kind = d.x & 3, n = (d.x >> 2) & 31;
            if (kind == EL_SKIP) continue;
            if (lane == 0) {
                sl_kind[warp][sl] = kind;
                sl_n[warp][sl] = n;
                sl_id[warp][sl] = d.y;
                sl_p[warp][sl] = 1 << ((d.x >> 7) & 3);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                if (kind == EL_Q) {
                    mbar_expect_tx(bar, (uint32_t)d.w);
                    bulk_g2s(dst, D.lg_pool + ((int64_t)(uint32_t)d.z << 9), (uint32_t)d.w, bar, l2_stream);
                } else {
                    mbar_expect_tx(bar, (uint32_t)kSlot);
                    tma_4d(dst, &tmap, 0, d.w, 0, d.z, bar, l2_stream);
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
    // ---- query B fragments. Column g of the N dimension is head g (G > 4) or
    // head g mod 4 (G <= 4); columns without a head hold zeros.
    const int hq_col = kDup ? (g & 3) : g;
    const bool col_ok = hq_col < G;
    const uint32_t *qw =
        reinterpret_cast<const uint32_t *>(q + ((int64_t)b * Hq + kvh * G + (col_ok ? hq_col : 0)) * kHeadDim);
    float qsum[kGroups] = {0.f, 0.f, 0.f, 0.f};   // sum of q over each group (column g)
    float bsum[kGroups] = {0.f, 0.f, 0.f, 0.f};   // sum of the INT2-path fragment values over each group
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        uint32_t lo = 0, hi = 0;   // channels (16ks+2t, +1) and (16ks+2t+8, +9)
        if (col_ok) {
            lo = qw[8 * ks + t];
            hi = qw[8 * ks + t + 4];
        }
        const float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&lo));
        const float2 c = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&hi));
        // INT2 path: k rows 2t, 2t+1 carry channels 2t, 2t+8 (they meet 128 + code);
        // k rows 2t+8, 2t+9 carry channels 2t+1, 2t+9 divided by 4 (they meet 128 + 4 code)
        const uint32_t x0 = (lo & 0xffffu) | (hi << 16);
        const uint32_t x1 = pack_rn(a.y * 0.25f, c.y * 0.25f);
        if (warp == 0) {
            s_qf[ks * 32 + lane] = make_uint2(lo, hi);
            s_qf[(8 + ks) * 32 + lane] = make_uint2(x0, x1);
        }
        qsum[ks >> 1] += (a.x + a.y) + (c.x + c.y);
        bsum[ks >> 1] += (a.x + c.x) + (bf_lo(x1) + bf_hi(x1));
    }
    // INT2 accumulator start per group: -128 x the fragment sum of columns 2t, 2t+1 (s_qb[grp][t])
    float qsel = 0.f;
#pragma unroll
    for (int i = 0; i < kGroups; ++i) {
        qsum[i] += __shfl_xor_sync(0xffffffffu, qsum[i], 1);
        qsum[i] += __shfl_xor_sync(0xffffffffu, qsum[i], 2);
        bsum[i] += __shfl_xor_sync(0xffffffffu, bsum[i], 1);
        bsum[i] += __shfl_xor_sync(0xffffffffu, bsum[i], 2);
        const float b0 = -128.f * __shfl_sync(0xffffffffu, bsum[i], 8 * t);
        const float b1 = -128.f * __shfl_sync(0xffffffffu, bsum[i], 8 * t + 4);
        if (warp == 0 && g == 0) s_qb[i * 4 + t] = make_float2(b0, b1);
        if (i == t) qsel = qsum[i];
    }
    // min-term B fragment: k rows 2t, 2t+1 = (hi, lo) fp16 parts of column g's group-t query sum
    uint32_t qs_frag;
    {
        const __half h = __float2half_rn(qsel);
        const __half l = __float2half_rn(qsel - __half2float(h));
        const __half2 p = __halves2half2(h, l);
        qs_frag = *reinterpret_cast<const uint32_t *>(&p);
    }
    __syncthreads();
    const float qk_scale = kLog2e * rsqrtf((float)kHeadDim);

    // ---- per-warp online softmax state, per N column (2t, 2t + 1 for this lane)
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, w0 = 0.f, w1 = 0.f;
    float o[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float mn0[kGroups] = {0.f, 0.f, 0.f, 0.f}, mn1[kGroups] = {0.f, 0.f, 0.f, 0.f};   // V minimum shares
    const float lo_f = t >= 2 ? 1.f : 0.f;   // with kDup: columns 4..7 (lanes t = 2, 3) take the lo parts of P
    // ldmatrix row addressing (full-precision tiles): token and 8-channel half of this lane's row
    const int lm_tok = ((lane >> 4) << 3) + (lane & 7);
    const int lm_hi = (lane >> 3) & 1;
    // the tokens of rows g and g + 8 in a quantised tile
    // the bf16 offset pattern of the code operands, in a register (Hq >> 31 is 0)
    const uint32_t k43 = 0x43004300u | ((uint32_t)Hq >> 31);
    const int tA = (g & 1) ? g + 7 : g;
    const int tB = (g & 1) ? g + 8 : g + 1;

    // softmax of the unscaled logits x = {(row g, col 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)}
    // in place; the scale (log2 e / sqrt(d)) joins each subtraction of the running max
    auto softmax = [&](float (&x)[4]) {
        const float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
        if (__any_sync(0xffffffffu, fmaf(mx0, qk_scale, -m0) > kLazy || fmaf(mx1, qk_scale, -m1) > kLazy)) {
            float h0 = mx0, h1 = mx1;
#pragma unroll
            for (int o2 = 4; o2 <= 16; o2 <<= 1) {
                h0 = fmaxf(h0, __shfl_xor_sync(0xffffffffu, h0, o2));
                h1 = fmaxf(h1, __shfl_xor_sync(0xffffffffu, h1, o2));
            }
            const float n0 = fmaxf(m0, h0 * qk_scale), n1 = fmaxf(m1, h1 * qk_scale);
            const float a0 = ex2(m0 - n0), a1 = ex2(m1 - n1);
            m0 = n0;
            m1 = n1;
            l0 *= a0;
            w0 *= a0;
            l1 *= a1;
            w1 *= a1;
#pragma unroll
            for (int i = 0; i < kGroups; ++i) {
                mn0[i] *= a0;
                mn1[i] *= a1;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                o[i][0] *= a0;
                o[i][1] *= a1;
                o[i][2] *= a0;
                o[i][3] *= a1;
            }
        }
        x[0] = ex2(fmaf(x[0], qk_scale, -m0));
        x[1] = ex2(fmaf(x[1], qk_scale, -m1));
        x[2] = ex2(fmaf(x[2], qk_scale, -m0));
        x[3] = ex2(fmaf(x[3], qk_scale, -m1));
        w0 += x[0] + x[2];
        w1 += x[1] + x[3];
    };
    // (reference max, exp-sum) per head of the chunk just finished, in the record slot
    // of its first tile; the slots of its other ntile - 1 tiles get empty records
    auto write_record = [&](int idx, int ntile) {
        float s0 = w0, s1 = w1;
#pragma unroll
        for (int o2 = 4; o2 <= 16; o2 <<= 1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, o2);
            s1 += __shfl_xor_sync(0xffffffffu, s1, o2);
        }
        if (g == 0) {
            float2 *r = rec + (int64_t)idx * G;
            if (2 * t < G) r[2 * t] = make_float2(m0, s0);
            if (2 * t + 1 < G) r[2 * t + 1] = make_float2(m1, s1);
        }
        for (int i = lane; i < (ntile - 1) * G; i += 32) rec[(int64_t)(idx + 1) * G + i] = make_float2(-INFINITY, 0.f);
        l0 += w0;
        l1 += w1;
        w0 = w1 = 0.f;
    };
    // P operand of the PV product from x (rows g, g + 8): X0 = rows 0-7, X1 = rows 8-15
    auto p_operand = [&](float p0, float p1, float p2, float p3, uint32_t &b0, uint32_t &b1, uint32_t &b2,
                         uint32_t &b3) {
        if (kDup) {
            b0 = movm_t(split_sel(p0, p1, lo_f));
            b1 = movm_t(split_sel(p2, p3, lo_f));
        } else {
            uint32_t h0, e0, h1, e1;
            split_pair(p0, p1, h0, e0);
            split_pair(p2, p3, h1, e1);
            b0 = movm_t(h0);
            b1 = movm_t(h1);
            b2 = movm_t(e0);
            b3 = movm_t(e1);
        }
    };
    auto pv_mma = [&](float (&acc)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                      uint32_t b1, uint32_t b2, uint32_t b3) {
        mma(acc, a0, a1, a2, a3, b0, b1);
        if (!kDup) mma(acc, a0, a1, a2, a3, b2, b3);
    };

    // ---- one quantised 16-token tile at `base` with P code planes. Pc is the plane
    // count, an int or a compile-time constant (PlanesC: the arithmetic of that width
    // alone); kch_tile: a K-channel tile (K groups of their own widths ahead of the
    // K meta, kcodes bytes)
    auto quant_tile = [&](const uint8_t *base, auto Pc, bool kch_tile) {
        const int P = static_cast<int>(Pc);
        const int kcodes = (kWide && kch_tile) ? s_kg[8] : -1;
        const uint8_t *km = base + (kcodes >= 0 ? kcodes : qtile_kmeta(P));
        const uint8_t *vc = base + (kcodes >= 0 ? kcodes + 256 : qtile_vcodes(P));
        const uint8_t *vm = base + (kcodes >= 0 ? kcodes + 256 + 512 * P : qtile_vmeta(P));
        // minimum share: one fp16 MMA; A rows g / g + 8 hold the tokens' group-t minimums twice
        float x[4];
        {
            const uint32_t mA = ld32(km + tA * 16 + t * 4), mB = ld32(km + tB * 16 + t * 4);
            mma_f16_k8(x, __byte_perm(mA, 0, 0x3232), __byte_perm(mB, 0, 0x3232), qs_frag);
        }
        const uint4 kmA = ld128(km + tA * 16), kmB = ld128(km + tB * 16);
        if (kWide && kcodes >= 0) {
            // K-channel tile: group grp has Pg planes of [16 tokens][8 B] at its offset;
            // a group of width 0 takes no part (its minimum is 0 in the meta as well)
#pragma unroll
            for (int grp = 0; grp < kGroups; ++grp) {
                const int Pg = s_kg[grp];
                if (Pg == 0) continue;
                const uint8_t *gb = base + s_kg[4 + grp];
                const float sA = h2f(pick(kmA, grp)).x, sB = h2f(pick(kmB, grp)).x;
                if (Pg == 1 || Pg == 2) {
                    float acc[4];
                    const uint2 a0 = ld64(gb + tA * 8), b0 = ld64(gb + tB * 8);
                    uint2 a1 = a0, b1 = b0;
                    if (Pg == 2) {
                        a1 = ld64(gb + 128 + tA * 8);
                        b1 = ld64(gb + 128 + tB * 8);
                    }
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const int ks = 2 * grp + kk;
                        const uint32_t xa = (kk ? a0.y : a0.x) >> (4 * t), xb = (kk ? b0.y : b0.x) >> (4 * t);
                        const uint32_t ya = (kk ? a1.y : a1.x) >> (4 * t), yb = (kk ? b1.y : b1.x) >> (4 * t);
                        const uint32_t c0 = Pg == 1 ? off_lo(xa, k43) : off4_lo(xa, ya, k43);
                        const uint32_t c1 = Pg == 1 ? off_lo(xb, k43) : off4_lo(xb, yb, k43);
                        const uint32_t c2 = Pg == 1 ? off_hi(xa, k43) : off4_hi(xa, ya, k43);
                        const uint32_t c3 = Pg == 1 ? off_hi(xb, k43) : off4_hi(xb, yb, k43);
                        const uint2 bq = s_qf[(8 + ks) * 32 + lane];
                        if (kk == 0) {
                            const float2 qb = s_qb[grp * 4 + t];
                            mma_c(acc, c0, c1, c2, c3, bq.x, bq.y, qb.x, qb.y);
                        } else {
                            mma(acc, c0, c1, c2, c3, bq.x, bq.y);
                        }
                    }
                    x[0] = fmaf(sA, acc[0], x[0]);
                    x[1] = fmaf(sA, acc[1], x[1]);
                    x[2] = fmaf(sB, acc[2], x[2]);
                    x[3] = fmaf(sB, acc[3], x[3]);
                } else {
                    // 8 bits: nibbles n0 = c0 + 4 c1 (planes 0, 1), n1 = c2 + 4 c3 (planes 2, 3)
                    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc16[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int pp = 0; pp < 2; ++pp) {
                        const uint8_t *kp = gb + 256 * pp;
                        const uint2 a0w = ld64(kp + tA * 8), a1w = ld64(kp + 128 + tA * 8);
                        const uint2 b0w = ld64(kp + tB * 8), b1w = ld64(kp + 128 + tB * 8);
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const int ks = 2 * grp + kk;
                            const uint32_t xa = (kk ? a0w.y : a0w.x) >> (4 * t), ya = (kk ? a1w.y : a1w.x) >> (4 * t);
                            const uint32_t xb = (kk ? b0w.y : b0w.x) >> (4 * t), yb = (kk ? b1w.y : b1w.x) >> (4 * t);
                            const uint2 bq = s_qf[(8 + ks) * 32 + lane];
                            const uint32_t c0 = bsub128(off4_lo(xa, ya, k43)), c1 = bsub128(off4_lo(xb, yb, k43));
                            const uint32_t c2 = bsub128(off4_hi(xa, ya, k43)), c3 = bsub128(off4_hi(xb, yb, k43));
                            if (pp == 0)
                                mma(acc, c0, c1, c2, c3, bq.x, bq.y);
                            else
                                mma(acc16, c0, c1, c2, c3, bq.x, bq.y);
                        }
                    }
                    x[0] = fmaf(sA, fmaf(16.f, acc16[0], acc[0]), x[0]);
                    x[1] = fmaf(sA, fmaf(16.f, acc16[1], acc[1]), x[1]);
                    x[2] = fmaf(sB, fmaf(16.f, acc16[2], acc[2]), x[2]);
                    x[3] = fmaf(sB, fmaf(16.f, acc16[3], acc[3]), x[3]);
                }
            }
        } else if (!kWide || P == 1) {
            const uint4 kA0 = ld128(base + tA * 32), kA1 = ld128(base + tA * 32 + 16);
            const uint4 kB0 = ld128(base + tB * 32), kB1 = ld128(base + tB * 32 + 16);
#pragma unroll
            for (int grp = 0; grp < kGroups; ++grp) {
                float acc[4];
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const int ks = 2 * grp + kk;
                    const uint32_t xa = pick(ks < 4 ? kA0 : kA1, ks & 3) >> (4 * t);
                    const uint32_t xb = pick(ks < 4 ? kB0 : kB1, ks & 3) >> (4 * t);
                    const uint2 bq = s_qf[(8 + ks) * 32 + lane];
                    if (kk == 0) {
                        const float2 qb = s_qb[grp * 4 + t];
                        mma_c(acc, off_lo(xa, k43), off_lo(xb, k43), off_hi(xa, k43), off_hi(xb, k43), bq.x, bq.y,
                              qb.x, qb.y);
                    }
                    else
                        mma(acc, off_lo(xa, k43), off_lo(xb, k43), off_hi(xa, k43), off_hi(xb, k43), bq.x, bq.y);
                }
                const float sA = h2f(pick(kmA, grp)).x, sB = h2f(pick(kmB, grp)).x;
                x[0] = fmaf(sA, acc[0], x[0]);
                x[1] = fmaf(sA, acc[1], x[1]);
                x[2] = fmaf(sB, acc[2], x[2]);
                x[3] = fmaf(sB, acc[3], x[3]);
            }
        } else if (P == 2) {
            // INT4: the two planes joined in registers into 4-bit codes, then the INT2 arithmetic
            const uint4 kA0 = ld128(base + tA * 32), kA1 = ld128(base + tA * 32 + 16);
            const uint4 kB0 = ld128(base + tB * 32), kB1 = ld128(base + tB * 32 + 16);
            const uint4 kA0p = ld128(base + 512 + tA * 32), kA1p = ld128(base + 512 + tA * 32 + 16);
            const uint4 kB0p = ld128(base + 512 + tB * 32), kB1p = ld128(base + 512 + tB * 32 + 16);
#pragma unroll
            for (int grp = 0; grp < kGroups; ++grp) {
                float acc[4];
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const int ks = 2 * grp + kk;
                    const uint32_t xa = pick(ks < 4 ? kA0 : kA1, ks & 3) >> (4 * t);
                    const uint32_t xb = pick(ks < 4 ? kB0 : kB1, ks & 3) >> (4 * t);
                    const uint32_t ya = pick(ks < 4 ? kA0p : kA1p, ks & 3) >> (4 * t);
                    const uint32_t yb = pick(ks < 4 ? kB0p : kB1p, ks & 3) >> (4 * t);
                    const uint2 bq = s_qf[(8 + ks) * 32 + lane];
                    if (kk == 0) {
                        const float2 qb = s_qb[grp * 4 + t];
                        mma_c(acc, off4_lo(xa, ya, k43), off4_lo(xb, yb, k43), off4_hi(xa, ya, k43),
                              off4_hi(xb, yb, k43), bq.x, bq.y, qb.x, qb.y);
                    }
                    else
                        mma(acc, off4_lo(xa, ya, k43), off4_lo(xb, yb, k43), off4_hi(xa, ya, k43),
                            off4_hi(xb, yb, k43), bq.x, bq.y);
                }
                const float sA = h2f(pick(kmA, grp)).x, sB = h2f(pick(kmB, grp)).x;
                x[0] = fmaf(sA, acc[0], x[0]);
                x[1] = fmaf(sA, acc[1], x[1]);
                x[2] = fmaf(sB, acc[2], x[2]);
                x[3] = fmaf(sB, acc[3], x[3]);
            }
        } else {
            // INT8: code = n0 + 16 n1 with nibbles n0 = c0 + 4 c1, n1 = c2 + 4 c3; each nibble
            // goes through the arithmetic with exact codes (offset removed), the high one weighted 16
#pragma unroll
            for (int grp = 0; grp < kGroups; ++grp) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc16[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int pp = 0; pp < 2; ++pp) {
                    const uint8_t *kp = base + 1024 * pp + grp * 8;
                    const uint2 a0w = ld64(kp + tA * 32), a1w = ld64(kp + 512 + tA * 32);
                    const uint2 b0w = ld64(kp + tB * 32), b1w = ld64(kp + 512 + tB * 32);
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const int ks = 2 * grp + kk;
                        const uint32_t xa = (kk ? a0w.y : a0w.x) >> (4 * t), ya = (kk ? a1w.y : a1w.x) >> (4 * t);
                        const uint32_t xb = (kk ? b0w.y : b0w.x) >> (4 * t), yb = (kk ? b1w.y : b1w.x) >> (4 * t);
                        const uint2 bq = s_qf[(8 + ks) * 32 + lane];
                        const uint32_t c0 = bsub128(off4_lo(xa, ya, k43)), c1 = bsub128(off4_lo(xb, yb, k43));
                        const uint32_t c2 = bsub128(off4_hi(xa, ya, k43)), c3 = bsub128(off4_hi(xb, yb, k43));
                        if (pp == 0)
                            mma(acc, c0, c1, c2, c3, bq.x, bq.y);
                        else
                            mma(acc16, c0, c1, c2, c3, bq.x, bq.y);
                    }
                }
                const float sA = h2f(pick(kmA, grp)).x, sB = h2f(pick(kmB, grp)).x;
                x[0] = fmaf(sA, fmaf(16.f, acc16[0], acc[0]), x[0]);
                x[1] = fmaf(sA, fmaf(16.f, acc16[1], acc[1]), x[1]);
                x[2] = fmaf(sB, fmaf(16.f, acc16[2], acc[2]), x[2]);
                x[3] = fmaf(sB, fmaf(16.f, acc16[3], acc[3]), x[3]);
            }
        }
        softmax(x);
        // ---- PV. Rows g + 8 (k rows 8-15 of the operand) meet 4 x code, so their P
        // parts carry the V scale divided by 4 (exact).
        const uint4 vmA = ld128(vm + tA * 16), vmB = ld128(vm + tB * 16);
#pragma unroll
        for (int grp = 0; grp < kGroups; ++grp) {
            const float2 fa = h2f(pick(vmA, grp)), fb = h2f(pick(vmB, grp));   // .x scale, .y min
            mn0[grp] = fmaf(x[0], fa.y, fmaf(x[2], fb.y, mn0[grp]));
            mn1[grp] = fmaf(x[1], fa.y, fmaf(x[3], fb.y, mn1[grp]));
            const float sb4 = 0.25f * fb.x;
            uint32_t b0, b1, b2 = 0, b3 = 0;
            p_operand(x[0] * fa.x, x[1] * fa.x, x[2] * sb4, x[3] * sb4, b0, b1, b2, b3);
            // words of this lane's channels: mt = 2 grp + mm; channel 16 mt + g (h = 0) and + 8 (h = 1)
            if (!kWide || P == 1) {
                const uint4 vv = ld128(vc + g * 64 + grp * 16);
#pragma unroll
                for (int mm = 0; mm < 2; ++mm) {
                    const uint32_t x0 = pick(vv, 2 * mm) >> (4 * t), x1 = pick(vv, 2 * mm + 1) >> (4 * t);
                    pv_mma(o[2 * grp + mm], bsub128(off_lo(x0, k43)), bsub128(off_lo(x1, k43)),
                           bsub128(off_hi(x0, k43)), bsub128(off_hi(x1, k43)), b0, b1, b2, b3);
                }
            } else if (P == 2) {
                const uint4 vv = ld128(vc + g * 64 + grp * 16), vp = ld128(vc + 512 + g * 64 + grp * 16);
#pragma unroll
                for (int mm = 0; mm < 2; ++mm) {
                    const uint32_t x0 = pick(vv, 2 * mm) >> (4 * t), x1 = pick(vv, 2 * mm + 1) >> (4 * t);
                    const uint32_t y0 = pick(vp, 2 * mm) >> (4 * t), y1 = pick(vp, 2 * mm + 1) >> (4 * t);
                    pv_mma(o[2 * grp + mm], bsub128(off4_lo(x0, y0, k43)), bsub128(off4_lo(x1, y1, k43)),
                           bsub128(off4_hi(x0, y0, k43)), bsub128(off4_hi(x1, y1, k43)), b0, b1, b2, b3);
                }
            } else {
#pragma unroll
                for (int pp = 0; pp < 2; ++pp) {
                    const uint4 vv = ld128(vc + 1024 * pp + g * 64 + grp * 16);
                    const uint4 vp = ld128(vc + 1024 * pp + 512 + g * 64 + grp * 16);
                    const uint32_t c0 = pp ? bmul16(b0) : b0, c1 = pp ? bmul16(b1) : b1;
                    const uint32_t c2 = pp ? bmul16(b2) : b2, c3 = pp ? bmul16(b3) : b3;
#pragma unroll
                    for (int mm = 0; mm < 2; ++mm) {
                        const uint32_t x0 = pick(vv, 2 * mm) >> (4 * t), x1 = pick(vv, 2 * mm + 1) >> (4 * t);
                        const uint32_t y0 = pick(vp, 2 * mm) >> (4 * t), y1 = pick(vp, 2 * mm + 1) >> (4 * t);
                        pv_mma(o[2 * grp + mm], bsub128(off4_lo(x0, y0, k43)), bsub128(off4_lo(x1, y1, k43)),
                               bsub128(off4_hi(x0, y0, k43)), bsub128(off4_hi(x1, y1, k43)), c0, c1, c2, c3);
                    }
                }
            }
        }
    };

    // ---- main loop
    while (consumed < issued) {
        const int sl = consumed % kSlots;
        const bool ok = mbar_wait(smem_u32(&bars[warp][sl]), (uint32_t)((consumed / kSlots) & 1));
        if (__any_sync(0xffffffffu, !ok)) {
            if (lane == 0) {
                set_status(C, QEVICT_ERR_TIMEOUT, layer, b, consumed);
                for (int r = consumed + 1; r < issued; ++r)
                    (void)mbar_wait(smem_u32(&bars[warp][r % kSlots]), (uint32_t)((r / kSlots) & 1));
            }
            break;
        }
        __syncwarp();
        const int kind = sl_kind[warp][sl], n = sl_n[warp][sl], id = sl_id[warp][sl];
        const uint32_t base = ring_s + sl * kSlot;
        if (kind == EL_Q) {
            const int P = kWide ? sl_p[warp][sl] : 1;
            const int tb = kWide ? qtile_bytes(P) : kQTile;
            const uint8_t *tp = smem + warp * kRing + sl * kSlot;
            // the tile arithmetic compiled for each plane count (K-channel tiles: generic)
            if (!kWide || (P == 1 && s_kg[8] < 0)) {
                for (int u = 0; u < n; ++u) quant_tile(tp + u * tb, PlanesC<1>{}, false);
            } else if (s_kg[8] >= 0) {
                for (int u = 0; u < n; ++u) quant_tile(tp + u * tb, P, true);
            } else if (P == 2) {
                for (int u = 0; u < n; ++u) quant_tile(tp + u * tb, PlanesC<2>{}, false);
            } else {
                for (int u = 0; u < n; ++u) quant_tile(tp + u * tb, PlanesC<4>{}, false);
            }
            write_record(id, n);
        } else if (kind == EL_F) {
            // ---------------- full-precision unit: QK, softmax, PV
            float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int chunk = 2 * (ks & 3) + lm_hi;
                const uint32_t addr = base + (ks >> 2) * 2048 + lm_tok * 128 + ((chunk ^ (lm_tok & 7)) << 4);
                uint32_t r0, r1, r2, r3;
                ldsm_x4(addr, r0, r1, r2, r3);
                const uint2 bq = s_qf[ks * 32 + lane];
                mma(x, r0, r2, r1, r3, bq.x, bq.y);
            }
            if (n < 16) {
                // rows past the open window's last token: P is 0 there, but the V rows
                // hold stale slot memory and 0 * NaN would still poison the product
                if (g >= n) x[0] = x[1] = -INFINITY;
                if (g + 8 >= n) x[2] = x[3] = -INFINITY;
                for (int cc = lane; cc < (16 - n) * 16; cc += 32) {
                    const int row = n + (cc >> 4), half = (cc >> 3) & 1, ch = cc & 7;
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(base + 4096 + half * 2048 +
                                                                                  row * 128 + ch * 16),
                                 "r"(0u)
                                 : "memory");
                }
                __syncwarp();
            }
            softmax(x);
            uint32_t b0, b1, b2 = 0, b3 = 0;
            p_operand(x[0], x[1], x[2], x[3], b0, b1, b2, b3);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const int chunk = 2 * (mt & 3) + lm_hi;
                const uint32_t addr = base + 4096 + (mt >> 2) * 2048 + lm_tok * 128 + ((chunk ^ (lm_tok & 7)) << 4);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(addr, a0, a1, a2, a3);
                pv_mma(o[mt], a0, a1, a2, a3, b0, b1, b2, b3);
            }
            write_record(id, 1);
        }
        __syncwarp();
        ++consumed;
        try_issue();
    }
    __syncthreads();

    // ---- merge the warps (the rings are free now); rows padded by 4 floats
    constexpr int kOwStride = kHeadDim + 4;
    float *Ow = reinterpret_cast<float *>(smem);    // [warp][8 columns][kOwStride]
    float *mw_s = Ow + kWarps * 8 * kOwStride;      // [warp][8] running max
    float *lw_s = mw_s + kWarps * 8;                // [warp][8] exp-sum
    float *fw_s = lw_s + kWarps * 8;                // [warp][8] weight of the warp in the split
    float *Mh_s = fw_s + kWarps * 8;                // [8] the split's max per head
#pragma unroll
    for (int o2 = 4; o2 <= 16; o2 <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o2);
#pragma unroll
        for (int i = 0; i < kGroups; ++i) {
            mn0[i] += __shfl_xor_sync(0xffffffffu, mn0[i], o2);
            mn1[i] += __shfl_xor_sync(0xffffffffu, mn1[i], o2);
        }
    }
    {
        // every N column as it is (with kDup, columns 4..7 hold the lo parts of columns
        // 0..3 and take no V minimum share); the minimum share joins its group's channels
        const int c0 = 2 * t, c1 = 2 * t + 1;
        const float mk = (kDup && t >= 2) ? 0.f : 1.f;
        float *ob = Ow + warp * 8 * kOwStride;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const float a0 = mk * mn0[mt >> 1], a1 = mk * mn1[mt >> 1];
            ob[c0 * kOwStride + 16 * mt + g] = o[mt][0] + a0;
            ob[c0 * kOwStride + 16 * mt + g + 8] = o[mt][2] + a0;
            ob[c1 * kOwStride + 16 * mt + g] = o[mt][1] + a1;
            ob[c1 * kOwStride + 16 * mt + g + 8] = o[mt][3] + a1;
        }
        if (g == 0) {
            mw_s[warp * 8 + c0] = m0;
            lw_s[warp * 8 + c0] = l0;
            mw_s[warp * 8 + c1] = m1;
            lw_s[warp * 8 + c1] = l1;
        }
    }
    __syncthreads();
    if (tid < kWarps * 8) {
        // the weight of warp ww in head hh's split result: 2^(m_ww - M)
        const int ww = tid >> 3, hh = tid & 7;
        float M = -INFINITY;
#pragma unroll
        for (int v = 0; v < kWarps; ++v) M = fmaxf(M, mw_s[v * 8 + hh]);
        fw_s[tid] = M == -INFINITY ? 0.f : ex2(mw_s[tid] - M);
        if (ww == 0) Mh_s[hh] = M;
    }
    __syncthreads();
    // ---- this split's partial output [G][128] (unnormalised, relative to its own
    // max) and (max, exp-sum) per head. Every value another split reads leaves as a
    // 64-bit word whose high half is this launch's tag, so a reader tells a current
    // value from a stale one by itself and no fence is needed.
    const uint32_t tag = s_gen + 1u;
    {
        unsigned long long *pw = S.part + ((int64_t)bk * splits + split) * G * kHeadDim;
        for (int i = tid; i < G * kHeadDim; i += kThreads) {
            const int hh = i / kHeadDim, c = i % kHeadDim;
            float acc = 0.f;
#pragma unroll
            for (int ww = 0; ww < kWarps; ++ww) {
                float v = Ow[(ww * 8 + hh) * kOwStride + c];
                if (kDup) v += Ow[(ww * 8 + hh + 4) * kOwStride + c];
                acc = fmaf(fw_s[ww * 8 + hh], v, acc);
            }
            const unsigned long long word = ((unsigned long long)tag << 32) | __float_as_uint(acc);
            asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(pw + i), "l"(word) : "memory");
            if (c == 0) {
                float l = 0.f;
#pragma unroll
                for (int ww = 0; ww < kWarps; ++ww) l = fmaf(fw_s[ww * 8 + hh], lw_s[ww * 8 + hh], l);
                unsigned long long *r = S.stat + (((int64_t)bk * kMaxSplits + split) * kMaxG + hh) * 2;
                const unsigned long long m64 = ((unsigned long long)tag << 32) | __float_as_uint(Mh_s[hh]);
                const unsigned long long l64 = ((unsigned long long)tag << 32) | __float_as_uint(l);
                asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(r), "l"(m64), "l"(l64) : "memory");
            }
        }
    }
    __syncthreads();   // this CTA's chunk records are in global memory; the shared buffers are free again
    if (knew != nullptr && tid == kThreads - 32) {
        // every table read of this CTA is behind it (the release orders them before the count)
        asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(S.arrive_b + b), "r"(1u) : "memory");
    }

    // ---- the tail: the splits meet, then each writes a slice of the output and the
    // masses of its own windows
    float *hM = reinterpret_cast<float *>(smem);    // [8] max over the splits and the new token
    float *hIL = hM + 8;                            // [8] 1 / exp-sum
    float *hFN = hM + 16;                           // [8] the new token's weight
    float *Fs = hM + 32;                            // [kMaxSplits][8] weight of each split
    float *sV = hM + 32 + kMaxSplits * 8;           // [128] the new token's V row
    float4 *red = reinterpret_cast<float4 *>(hM + 2048);   // [slice outputs][splits]
    // the tables as this launch found them: once every CTA of the sequence has
    // published, one CTA moves them on, so nothing below reads them afresh
    const int64_t length = s_len;
    const bool has_new = knew != nullptr && length < D.max_context;
    if (knew != nullptr && !has_new && tid == 0 && split == 0)   // replayed past the end of the tables
        set_status(C, QEVICT_ERR_INVALID_ARG, layer, b, (int)length);
    const int64_t wb = (int64_t)b * D.Wmax;
    const int n_win = (int)((length + w - 1) / w);
    const int64_t Lnew = has_new ? length + 1 : length;
    const int n_out = (int)((Lnew + w - 1) / w);
    const int wnew = (int)(length / w);
    const bool opens = has_new && (length % w == 0);
    const __nv_bfloat16 *kn = has_new ? knew + ((int64_t)b * Hkv + kvh) * kHeadDim : nullptr;
    const __nv_bfloat16 *vn = has_new ? vnew + ((int64_t)b * Hkv + kvh) * kHeadDim : nullptr;
    const float inv_hq = 1.f / (float)Hq;
    float *sp = D.score_part + ((int64_t)b * Hkv + kvh) * D.Wmax;

    const int qw0 = s_span[0], nqw = s_span[1], fw0 = s_span[2], nfw = s_span[3];
    // this split's windows: thread kMassT0 + i takes window i of the split (its
    // records for every head are loaded now, before the splits meet)
    const int nwin_s = nqw + nfw;
    constexpr int kMassT0 = kThreads - 128;   // threads of the mass work
    const int mi = tid - kMassT0;
    constexpr int kRecLd = G * 4;   // records loaded ahead: four tiles' worth (the rest when used)
    float2 mrec[kRecLd];
    int mwi = -1, mr0 = 0;
    if (mi >= 0 && mi < nwin_s) {
        const bool isq = mi < nqw;
        const int e = isq ? qw0 + mi : fw0 + (mi - nqw);
        mr0 = isq ? (D.CF + e) * mu : e * mu;
        mwi = (isq ? D.q_list[b * D.CQ + e] : D.fp_list[b * D.CF + e]).x;
#pragma unroll
        for (int k = 0; k < kRecLd; ++k)
            mrec[k] = (k / G < mu) ? rec[(int64_t)mr0 * G + k] : make_float2(0.f, 0.f);
    }
    // and the window's partial score (no other CTA writes it in this launch)
    const float msp = (accumulate && mwi >= 0) ? sp[mwi] : 0.f;
    // the evicted windows of this split's slice of [0, n_out), and the window this step opens
    const int z0 = (int)((int64_t)split * n_out / splits), z1 = (int)((int64_t)(split + 1) * n_out / splits);
    const int zi = z0 + tid;
    const uint8_t ztier = zi < min(z1, n_win) ? D.tier[wb + zi] : (uint8_t)QEVICT_TIER_E;
    // the new token's inputs
    uint2 nq_raw = make_uint2(0u, 0u), nk_raw = make_uint2(0u, 0u);
    if (has_new && warp < G) {
        nq_raw = reinterpret_cast<const uint2 *>(q + ((int64_t)b * Hq + kvh * G + warp) * kHeadDim)[lane];
        nk_raw = reinterpret_cast<const uint2 *>(kn)[lane];
    }
    if (has_new && tid < kHeadDim) sV[tid] = __bfloat162float(vn[tid]);

    // ---- the splits meet: warp hh polls head hh's (max, exp-sum) records, lane = split
    // (bounded: a wait that runs out sets TIMEOUT and takes the record as empty)
    if (warp < G) {
        const int hh = warp;
        float nl = -INFINITY;
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
            const unsigned long long *r = S.stat + (((int64_t)bk * kMaxSplits + lane) * kMaxG + hh) * 2;
            unsigned long long m64, l64;
            const long long t0 = clock64();
            while (true) {
                asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(m64), "=l"(l64) : "l"(r) : "memory");
                if ((uint32_t)(m64 >> 32) == tag && (uint32_t)(l64 >> 32) == tag) break;
                if (clock64() - t0 > C.wait_cycles) {
                    ok = false;
                    break;
                }
                __nanosleep(32);
            }
            if (ok) v = make_float2(__uint_as_float((uint32_t)m64), __uint_as_float((uint32_t)l64));
        }
        if (__any_sync(0xffffffffu, !ok) && lane == 0) set_status(C, QEVICT_ERR_TIMEOUT, layer, b, -3);
        float M = v.x;
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
        M = fmaxf(M, nl);
        const float f = (lane < splits && M != -INFINITY && v.x != -INFINITY) ? ex2(v.x - M) : 0.f;
        if (lane < splits) Fs[lane * 8 + hh] = f;
        float l = f * v.y;
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o2);
        if (lane == 0) {
            const float fn = has_new ? ex2(nl - M) : 0.f;
            l += fn;
            hM[hh] = M;
            hIL[hh] = l > 0.f ? 1.f / l : 0.f;
            hFN[hh] = fn;
        }
    }
    // ---- output gather: this split's slice of the [G][32] output float4s, one
    // (output, split) item per thread of the warps that do not poll, waiting until
    // the four tagged words of the item are current
    const int n4 = G * (kHeadDim / 4);
    const int o0 = split * n4 / splits, o1 = (split + 1) * n4 / splits;
    const int nwork = (o1 - o0) * splits;
    if (warp >= G) {
        const unsigned long long *pw = S.part + (int64_t)bk * splits * G * kHeadDim;
        bool ok = true;
        for (int it = tid - G * 32; it < nwork; it += kThreads - G * 32) {
            const int oi = o0 + it / splits, r = it % splits;
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
                if (clock64() - t0 > C.wait_cycles) {
                    ok = false;
                    break;
                }
                __nanosleep(32);
            }
            red[it] = ok ? make_float4(__uint_as_float((uint32_t)u0), __uint_as_float((uint32_t)u1),
                                       __uint_as_float((uint32_t)u2), __uint_as_float((uint32_t)u3))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (!ok) set_status(C, QEVICT_ERR_TIMEOUT, layer, b, -4);
    }
    __syncthreads();
    // output: the gathered partials weighted by their splits' factors
    for (int it = tid; it < o1 - o0; it += kThreads) {
        const int oi = o0 + it;
        const int hh = oi / (kHeadDim / 4), c4 = oi % (kHeadDim / 4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (has_new) {
            const float fn = hFN[hh];
            acc = make_float4(fn * sV[4 * c4], fn * sV[4 * c4 + 1], fn * sV[4 * c4 + 2], fn * sV[4 * c4 + 3]);
        }
        for (int r = 0; r < splits; ++r) {
            const float f = Fs[r * 8 + hh];
            const float4 v = red[it * splits + r];
            acc.x = fmaf(f, v.x, acc.x);
            acc.y = fmaf(f, v.y, acc.y);
            acc.z = fmaf(f, v.z, acc.z);
            acc.w = fmaf(f, v.w, acc.w);
        }
        const float il = hIL[hh];
        reinterpret_cast<float4 *>(out + ((int64_t)b * Hq + kvh * G + hh) * kHeadDim)[c4] =
            make_float4(acc.x * il, acc.y * il, acc.z * il, acc.w * il);
    }

    // ---- masses and cumulative scores of this split's windows: one thread per window
    // (the output threads above and the evicted sweep below run beside it)
    for (int wl = mi; mi >= 0 && wl < nwin_s; wl += 128) {
        int wi = mwi, r0 = mr0;
        if (wl != mi) {
            const bool isq = wl < nqw;
            const int e = isq ? qw0 + wl : fw0 + (wl - nqw);
            r0 = isq ? (D.CF + e) * mu : e * mu;
            wi = (isq ? D.q_list[b * D.CQ + e] : D.fp_list[b * D.CF + e]).x;
        }
        const bool isq = wl < nqw;
        const int nr = isq ? mu : ((wi == n_win - 1 ? (int)(length - (int64_t)wi * w) : w) + 15) >> 4;
        float sum = 0.f;
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            float m = 0.f;
            const float M = hM[hh];
            if (M != -INFINITY) {
#pragma unroll
                for (int r = 0; r < kRecMax; ++r) {
                    if (r >= nr) break;
                    const int k = r * G + hh;
                    const float2 st = (wl == mi && k < kRecLd) ? mrec[k < kRecLd ? k : 0] : rec[(int64_t)r0 * G + k];
                    if (st.y > 0.f) m = fmaf(st.y, ex2(st.x - M), m);
                }
                if (has_new && !opens && wi == wnew) m += hFN[hh];   // the new token joins the open window
                m *= hIL[hh];
            }
            if (mass) mass[((int64_t)b * Hq + kvh * G + hh) * n_out + wi] = m;
            sum += m;
        }
        if (accumulate) sp[wi] = (wl == mi ? msp : sp[wi]) + sum * inv_hq;
    }
    // windows no list holds, in this split's slice: evicted ones (mass 0) and the window this step opens
    for (int wi = zi; wi < z1; wi += kThreads) {
        const bool fresh = opens && wi == wnew;
        const uint8_t tr = wi == zi ? ztier : (wi < n_win ? D.tier[wb + wi] : (uint8_t)QEVICT_TIER_E);
        if (!fresh && (wi >= n_win || tr != QEVICT_TIER_E)) continue;
        float sum = 0.f;
#pragma unroll
        for (int h2 = 0; h2 < G; ++h2) {
            const float m = fresh ? hFN[h2] * hIL[h2] : 0.f;
            if (mass) mass[((int64_t)b * Hq + kvh * G + h2) * n_out + wi] = m;
            sum += m;
        }
        if (accumulate && fresh) atomicAdd(&sp[wi], sum * inv_hq);
    }
    // ---- the fused append (split 0): this KV head's K and V rows of the new token, into
    // the slot that receives it (read in the prologue, before this CTA's arrival: the
    // tables move on only after every CTA of the sequence has arrived)
    if (has_new && split == 0 && tid < 32) {
        const int slot_new = s_slot_new;
        if (slot_new >= 0) {
            const int row = (int)(length % w);
            const int kvs = tid >> 4, c = tid & 15;
            const __nv_bfloat16 *src = kvs ? vn : kn;
            __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(D.fp_pool + (int64_t)slot_new * D.fp_slot_bytes) +
                                 fp_off(kvh, kvs, w, row, 8 * c);
            *reinterpret_cast<uint4 *>(dst) = reinterpret_cast<const uint4 *>(src)[c];
        }
    }
    // The record generation moves on once per launch (split 0, after its meet: every
    // split of the pair has read it by then); the next launch reads it after its
    // dependency wait.
    if (split == 0 && tid == 0)
        asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(S.bar + 2 * bk + 1), "r"(1u) : "memory");
    // With a new token, split 0 of KV head 0 moves the sequence's tables on once every
    // CTA of the sequence has arrived (bounded wait): the length, and the window this
    // step opens with the next free slot.
    if (knew != nullptr && split == 0 && kvh == 0 && tid == 0) {
        const uint32_t want = (uint32_t)(Hkv * splits);
        uint32_t n = 0;
        const long long t0 = clock64();
        while (true) {
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(n) : "l"(S.arrive_b + b) : "memory");
            if (n >= want) break;
            if (clock64() - t0 > C.wait_cycles) break;
            __nanosleep(64);
        }
        if (n < want) {
            set_status(C, QEVICT_ERR_TIMEOUT, layer, b, -5);
        } else if (has_new) {
            S.arrive_b[b] = 0u;
            int32_t *c = D.ctr + b * kCtrN;
            if (opens) {
                const int n_fp = c[CTR_NFP];
                const int slotn = c[CTR_NEXT];
                if (slotn < 0) {
                    set_status(C, QEVICT_ERR_CAPACITY, layer, b, wnew);
                } else {
                    D.tier[wb + wnew] = QEVICT_TIER_FP;
                    D.fp_slot[wb + wnew] = slotn;
                    D.lg_slot[wb + wnew] = -1;
                    D.lwrites[wb + wnew] = 0;
                    D.fp_list[b * D.CF + n_fp] = make_int2(wnew, slotn);
                    c[CTR_NFP] = n_fp + 1;
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
        } else {
            S.arrive_b[b] = 0u;
        }
    }
}

constexpr int kDynSmem = kWarps * kRing + kDescTab * 16 + 16 * 32 * 8 + kGroups * 4 * 8 + 1024;

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

// Splits per (sequence, KV head): as many as fill the GPU in one wave, at
// most kMaxSplits.
int decode_splits(int pairs, int num_sms, int G) {
    const int per_sm = (G >= 1 && G <= kMaxG && g_ctas_per_sm[G] > 0) ? g_ctas_per_sm[G] : 1;
    int s = per_sm * num_sms / (pairs > 0 ? pairs : 1);
    if (s > kMaxSplits) s = kMaxSplits;
    if (s < 1) s = 1;
    return s;
}

// Records per (sequence, KV head): one per 16-token tile of every slot of the
// full-precision and the ledger pool.
int decode_records(int CF, int CQ, int w, int maxP) {
    (void)maxP;
    return (CF + CQ) * (w / 16);
}

cudaError_t launch_decode(const LayerDev &L, const CacheDev &C, const DecodeScratch &S, const CUtensorMap &tmap,
                          int layer, const __nv_bfloat16 *q, const __nv_bfloat16 *knew, const __nv_bfloat16 *vnew,
                          float *out, float *mass, int accumulate, int splits, bool pdl, bool coop,
                          cudaStream_t s) {
    const bool wide = L.maxP > 1;
    // The splits of a (sequence, KV head) wait for one another. A cooperative grid
    // starts only when every CTA can be resident at once, so another kernel holding
    // SMs delays the start instead of stranding a waiting split.
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (coop) {
        attr[na].id = cudaLaunchAttributeCooperative;
        attr[na].val.cooperative = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(splits, L.B * L.Hkv);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kDynSmem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = na;
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
