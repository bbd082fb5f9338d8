// Internal declarations shared by the translation units of the library:
// the device view of one layer, launch entry points, and small PTX helpers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/qevict.h"

namespace qevict {

constexpr int kHeadDim = 128;          // d
constexpr int kGroup = 32;             // channels per INT2 group
constexpr int kGroups = kHeadDim / kGroup;
constexpr int kMaxG = 8;               // query heads per KV head
constexpr int kMaxSplits = 32;         // decode CTAs per (sequence, KV head)
constexpr int kVTile = 16;             // tokens per transposed V-code word
constexpr int kCtrN = 16;              // counters per sequence

// counter slots (per sequence). CTR_NEXT is a full-precision slot taken off the
// free list ahead of time for the next window to open (-1 if none was free).
enum { CTR_NFP = 0, CTR_NQ = 1, CTR_FP_TOP = 2, CTR_LG_TOP = 3, CTR_WQ = 4, CTR_WP = 5,
       CTR_WC = 6, CTR_LEN = 7, CTR_NEXT = 8, CTR_KCH = 9 };
// CTR_KCH: 1 once qevict_route_rd_kv has set the sequence's K group widths (its
// quantised windows then hold K-channel tiles, see ktile_kcodes)

// device stats slots
enum { ST_DEMOTE = 0, ST_PROMOTE = 1, ST_EVICT = 2, ST_LWRITE = 3, ST_LREUSE = 4, ST_N = 8 };

// Full-precision slot: bf16 [Hkv][2 (K, V)][2 (channels 0-63, 64-127)][w][64].
// Element offset of channel c of token t of (KV head kvh, K or V).
__host__ __device__ inline int64_t fp_off(int kvh, int kv, int w, int t, int c) {
    return ((((int64_t)(kvh * 2 + kv) * 2 + (c >> 6)) * w + t) * 64) + (c & 63);
}

// Ledger slot: per KV head, w / 16 tiles of 16 tokens, each tile kQTile bytes:
// K codes [16][32 B] at 0, K meta [16][4] half2 at 512, V codes (128 words) at
// 768, V meta [16][4] half2 at 1280.
constexpr int kQTile = 1536;
constexpr int kTileKMeta = 512, kTileVCodes = 768, kTileVMeta = 1280;
__host__ __device__ inline int64_t lg_tile_off(int kvh, int w, int tile) {
    return ((int64_t)kvh * (w / 16) + tile) * kQTile;
}

// Wider codes (4 or 8 bits, P = bits / 2 planes): code = sum_p 4^p c_p with
// 2-bit planes c_p, each plane in the INT2 code layout. A tile holds the K
// planes at p * 512, the K meta after them, the V planes, then the V meta:
// 1024 P + 512 bytes; P = 1 is the INT2 tile above.
__host__ __device__ inline int qtile_bytes(int P) { return 1024 * P + 512; }
__host__ __device__ inline int qtile_kmeta(int P) { return 512 * P; }
__host__ __device__ inline int qtile_vcodes(int P) { return 512 * P + 256; }
__host__ __device__ inline int qtile_vmeta(int P) { return 1024 * P + 256; }
__host__ __device__ inline int64_t lg_tile_off(int kvh, int w, int tile, int P) {
    return ((int64_t)kvh * (w / 16) + tile) * qtile_bytes(P);
}
// A quantised window list entry's slot field: slot | log2(P) << 24 (0 for INT2).
constexpr int kSlotBits = 24;
__host__ __device__ inline bool is_quant_tier(int t) {
    return t == QEVICT_TIER_Q || t == QEVICT_TIER_Q4 || t == QEVICT_TIER_Q8;
}
__host__ __device__ inline int tier_bits(int t) {
    return t == QEVICT_TIER_Q4 ? 4 : (t == QEVICT_TIER_Q8 ? 8 : 2);
}

// V codes of a 16-token tile are 128 uint32 words, word i = (g * 8 + mt) * 2 + h
// holding channel 16 * mt + g + 8 * h (g, mt in 0..7, h in 0..1). This puts the
// 16 words one MMA lane group needs for the transposed-V operand side by side.
__host__ __device__ inline int vword_dim(int i) {
    const int g = i >> 4, mt = (i >> 1) & 7, h = i & 1;
    return 16 * mt + g + 8 * h;
}
__host__ __device__ inline int vword_index(int ch) {
    const int mt = ch >> 4, r = ch & 15, g = r & 7, h = r >> 3;
    return (g * 8 + mt) * 2 + h;
}

// Everything a kernel needs about one layer of the cache (passed by value).
struct LayerDev {
    int B, Hq, Hkv, G, w, Wmax, CF, CQ;   // per unit: a sequence, or a (sequence, KV head) pair
    int hs;                     // KV heads folded into units: 1, or the model's Hkv with per-head tiers
    int maxP;                   // planes of the widest ledger width allowed: 1 (INT2), 2 (INT4), 4 (INT8)
    int max_context;
    double beta, rho;           // budget fraction and its full-precision share
    int64_t c_fp, c_q;          // bytes of one window per sequence in each visible tier
    int64_t fp_slot_bytes, lg_slot_bytes;
    uint8_t *fp_pool;     // [B*CF][fp_slot_bytes]   see fp_off
    uint8_t *lg_pool;     // [B*CQ][lg_slot_bytes]   see lg_tile_off
    uint8_t *tier;        // [B][Wmax]
    int32_t *fp_slot;     // [B][Wmax]
    int32_t *lg_slot;     // [B][Wmax]
    int32_t *lwrites;     // [B][Wmax]
    float *score_part;    // [B][Hkv][Wmax] per-KV-head-group partial cumulative scores
    int32_t *fp_free;     // [B][CF] stack of free slot indices
    int32_t *lg_free;     // [B][CQ]
    int2 *fp_list;        // [B][CF] {window, slot} of full-precision windows
    int2 *q_list;         // [B][CQ] {window, slot} of INT2 windows
    int32_t *ctr;         // [B][kCtrN]; CTR_LEN is the context length the kernels use
    int4 *work_q;         // [B][Wmax] quantise: {window, src fp slot or -1 (external), dst ledger slot, 0}
    int4 *work_p;         // [B][Wmax] promote: {window, src ledger slot, dst fp slot, 0}
    int4 *work_c;         // [B][Wmax] prefill copy: {window, dst fp slot, 0, 0}
    int32_t *diag;        // [B][8] counts of the last completed tier move (see qevict_get_tier_move_counts)
    uint8_t *lbits;       // [B][Wmax] width of the window's ledger entry: 0 (none), 2, 4 or 8
    uint8_t *kgw;         // [B][Hkv][4] K group widths (0, 2, 4, 8) where ctr[CTR_KCH] is set
};

// K-channel ledger tile (a layer routed by qevict_route_rd_kv): per 16-token tile,
//   K codes of group g = 0..3 in turn: P_g planes (width / 2) of [16 tokens][8 B],
//   K meta [16][4] half2 (scale, minimum; zero for a group of width 0),
//   V codes (P_V planes of 512 B) and V meta (256 B) as in the plane tile.
// Tiles sit at the stride of the widest plane tile (qtile_bytes(4)).
__host__ __device__ inline int kgroup_planes(int bits) { return bits >> 1; }
__host__ __device__ inline int ktile_kcodes(const uint8_t *kw) {   // bytes of the K codes
    return 128 * (kgroup_planes(kw[0]) + kgroup_planes(kw[1]) + kgroup_planes(kw[2]) + kgroup_planes(kw[3]));
}
__host__ __device__ inline int ktile_bytes(int kcodes, int P) { return kcodes + 512 + 512 * P; }

// Row of token t of unit u in a caller's [units / hs][n][Hkv * hs][d] token array
// (a unit is a sequence, or with per-head tiers a (sequence, KV head) pair)
__device__ __forceinline__ int64_t src_row(const LayerDev &D, int u, int64_t n, int64_t t, int h) {
    return (((int64_t)(u / D.hs) * n + t) * D.hs + u % D.hs) * D.Hkv + h;
}

// Decode scratch, shared by all layers of a cache: a decode launch touches it
// only after its dependency wait, so consecutive launches never overlap in it.
struct DecodeScratch {
    unsigned long long *part;  // [B*Hkv][splits][G][d] split partial outputs (unnormalised, relative to the
                               // split's max): float in the low half, the launch's tag in the high half
    unsigned long long *stat;  // [B*Hkv][kMaxSplits][kMaxG][2] split (max, exp-sum), log2 domain, tagged likewise
    float2 *rec;          // [B*Hkv][rec_stride][G] (reference max, exp-sum) of each full-precision unit and
                          // quantised chunk, log2 domain (written and read by the same split)
    int rec_stride;       // records per (sequence, KV head): decode_records(CF, CQ, w, maxP)
    float2 *wstat;        // [B][Hq][max(Wmax, 2)] future-missed-mass partials
    uint32_t *bar;        // [B*Hkv][2] a counter of the missed-mass kernel (0 between launches), the
                          // decode's record generation
    uint32_t *arrive_b;   // [B] arrival counters of a sequence's CTAs for the fused append (0 between launches)
};

struct CacheDev {
    int32_t *status;              // [4]: code, layer, info0, info1
    unsigned long long *stats;    // [ST_N]
    long long wait_cycles;        // limit of a decode's waits on other CTAs (clock64 cycles)
};
constexpr long long kDefaultWaitCycles = 4000000000ll;   // about two seconds at GB300 clocks

enum PlanMode { PLAN_ROUTE = 0, PLAN_TIERS = 1, PLAN_PREFILL_SCORES = 2, PLAN_PREFILL_TIERS = 3,
                PLAN_DEMOTE = 4, PLAN_PROMOTE = 5, PLAN_GLOBAL = 6, PLAN_LOGSPARSE = 7, PLAN_RD = 8,
                PLAN_RD_MIXED = 9, PLAN_RD_KV = 10 };

struct PlanArgs {
    int mode;
    int layer;
    int64_t prefill_len;  // tokens a prefill brings (prefill modes only)
    const float *scores;  // override / prefill scores [B][n_win]
    const float *mult;    // [B][n_win]
    const uint8_t *tiers; // [B][n_win]
    const int32_t *pairs; // [n][2]
    int n_pairs;
    int recent;           // PLAN_LOGSPARSE: dense recent windows
    // PLAN_GLOBAL: the ranking keys and thresholds of one routing event over all layers
    const unsigned long long *gkeys;   // [sequences][layers][hs][Wmax], 0 for non-candidates
    const unsigned long long *gthr;    // [sequences][2]: keys >= [0] full precision, >= [1] INT2
    const int32_t *gflag;              // [sequences]: 0 = leave this sequence's tiers unchanged
    int glayers;                       // layers in the key table
    const float *kweights;             // PLAN_RD_KV: K channel weights [B][Hkv][d]
};

// One routing event over all layers of a cache under one budget per sequence.
struct GlobalArgs {
    const LayerDev *layers;            // device table [num_layers]
    int num_layers, hs, Wmax, w;
    double beta, rho;
    int64_t c_fp, c_q;                 // window costs of one unit
    unsigned long long *keys;          // as PlanArgs::gkeys
    unsigned long long *thr;
    int32_t *flag;
    int32_t *cnt;                      // [sequences][4]: candidates, forced, non-finite (0 between events)
};

// ---- launchers (each enqueues on `s`, returns the launch error) -----------
cudaError_t launch_init_layer(const LayerDev &L, cudaStream_t s);
// Keys (all layers in parallel), then budget, counts and the two thresholds of
// a global routing event (one CTA per sequence)
cudaError_t launch_global_select(const GlobalArgs &g, const CacheDev &C, int sequences, cudaStream_t s);
// Replace a layer's cumulative scores by scores [units][n_win] (the override of a global event)
cudaError_t launch_set_scores(const LayerDev &L, const float *scores, int n_win, cudaStream_t s);
cudaError_t launch_append(const LayerDev &L, const CacheDev &C, int layer, const __nv_bfloat16 *k,
                          const __nv_bfloat16 *v, int n_new, cudaStream_t s);
// Runs setup() once per (call site, key, current device) in the process, under
// a lock; a set-up that failed runs again on the next call. Kernel
// attributes such as the dynamic shared-memory limit belong to a device's
// context, so each device the library meets gets its own set-up.
constexpr int kOnceDevices = 64;
constexpr int kOnceKeys = 16;
template <class F>
inline cudaError_t once_per_device(int key, F &&setup) {
    static std::mutex mu;
    static bool done[kOnceKeys][kOnceDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= kOnceDevices || key < 0 || key >= kOnceKeys) return setup();
    if (done[key][dev]) return cudaSuccess;
    e = setup();
    if (e == cudaSuccess) done[key][dev] = true;
    return e;
}

cudaError_t launch_plan(const LayerDev &L, const CacheDev &C, const PlanArgs &a, cudaStream_t s);
cudaError_t launch_quantize(const LayerDev &L, const CacheDev &C, int layer, const __nv_bfloat16 *k_ext,
                            const __nv_bfloat16 *v_ext, int64_t ext_len, int max_entries,
                            cudaStream_t s);
cudaError_t launch_promote(const LayerDev &L, const CacheDev &C, int max_entries, cudaStream_t s);
cudaError_t launch_prefill_copy(const LayerDev &L, const __nv_bfloat16 *k_ext,
                                const __nv_bfloat16 *v_ext, int64_t ext_len, int max_entries,
                                cudaStream_t s);
cudaError_t launch_scores(const LayerDev &L, int n_win, float *out, cudaStream_t s);
cudaError_t launch_decode(const LayerDev &L, const CacheDev &C, const DecodeScratch &S, const CUtensorMap &tmap,
                          int layer, const __nv_bfloat16 *q, const __nv_bfloat16 *knew, const __nv_bfloat16 *vnew,
                          float *out, float *mass, int accumulate, int splits, bool pdl, bool coop,
                          cudaStream_t s);
cudaError_t launch_k_channel_weights(const LayerDev &L, const __nv_bfloat16 *q, int n_q, const __nv_bfloat16 *k,
                                     int64_t n_tok, float *out, cudaStream_t s);
cudaError_t launch_read_lengths(const LayerDev &L, int32_t *out, cudaStream_t s);
// kmap: k_full [sequences * n_tokens][Hkv * hs][128] bf16 as a 3-D tiled map,
// boxes of 64 channels x 1 KV head x 16 tokens, 128-byte swizzle
cudaError_t launch_future_missed_mass(const LayerDev &L, const CacheDev &C, const DecodeScratch &S, int layer,
                                      const CUtensorMap &kmap, const __nv_bfloat16 *q, int n_tokens, float *fmm,
                                      int num_sms, cudaStream_t s);
int decode_splits(int pairs, int num_sms, int G);
int decode_records(int CF, int CQ, int w, int maxP);
cudaError_t prepare_decode();

// ---- device helpers -------------------------------------------------------
__device__ __forceinline__ void set_status(const CacheDev &C, int code, int layer, int i0, int i1) {
    if (atomicCAS(C.status, 0, code) == 0) {
        C.status[1] = layer;
        C.status[2] = i0;
        C.status[3] = i1;
    }
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

}  // namespace qevict
