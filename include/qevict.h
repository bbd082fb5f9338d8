/*
 * qevict.h - C ABI of a GB300 (sm_103a) library for single-token GQA decode
 * attention over QEvict's recoverable three-tier KV cache.
 *
 * Method: "Technische Samenvatting: QEvict" (gist.science/nl/paper/2608.05326;
 * Chinese twin gist.science/zh/paper/2608.05326). Sections "Methodologie:
 * QEvict" (history split into consecutive windows, each kept in full precision,
 * in a recoverable INT2 tier, or evicted, inside one fixed byte budget) and
 * "Kernmechanismen" (window-level routing, cumulative attention scoring,
 * demotion, promotion, the write-once quantisation ledger, GQA support).
 * Evicted tokens leave the softmax normalisation ("Technische Samenvatting:
 * LogQuant", Methodologie 3) and the order of cache entries does not change
 * the attention output (same page, Methodologie 4), which lets the kernels
 * store and visit the tiers in any order.
 *
 * Conventions for every call:
 *  - Tensors are dense, row-major, on the device of the cache (device
 *    pointers) unless a parameter says "host". bf16 is IEEE bfloat16.
 *  - Every call that takes a `stream` (a cudaStream_t, NULL = legacy default
 *    stream) only enqueues work on it and returns without synchronising,
 *    except qevict_get_status / qevict_get_stats /
 *    qevict_get_tier_move_counts / qevict_refresh_lengths /
 *    qevict_cache_create / qevict_cache_destroy, which synchronise it.
 *  - Errors the host can see (bad arguments, a budget that cannot hold the
 *    open window, a full context) return a status at once and enqueue
 *    nothing; the cache is unchanged. Errors only the device can see (a
 *    slot pool running out, an illegal tier transition named by the caller,
 *    a non-finite score or K/V value, an fp16 overflow of the INT2 scale)
 *    set a sticky device status word, skip the offending work and are
 *    reported by qevict_get_status. No kernel traps or asserts.
 *  - Calls on one layer must be ordered (one stream, or events). Routing and
 *    tier moves of different layers may run concurrently on different
 *    streams: the shared status word and statistics are updated atomically.
 *    Calls that use the cache-wide decode scratch (the decode calls and
 *    qevict_future_missed_mass) must not overlap one another, nor may two
 *    qevict_route_global events. The host side is not thread-safe.
 *  - qevict_last_error() returns a thread-local message for the last host
 *    error of the calling thread.
 */
#ifndef QEVICT_H
#define QEVICT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum qevict_status {
    QEVICT_OK = 0,
    QEVICT_ERR_INVALID_ARG = 1,   /* a parameter is out of range or NULL */
    QEVICT_ERR_OUT_OF_MEMORY = 2, /* the allocator returned NULL */
    QEVICT_ERR_BUDGET = 3,        /* the byte budget cannot hold the open window */
    QEVICT_ERR_STATE = 4,         /* illegal tier transition / append into a non-FP window */
    QEVICT_ERR_CUDA = 5,          /* a CUDA runtime call failed */
    QEVICT_ERR_TIMEOUT = 6,       /* a bounded device wait gave up */
    QEVICT_ERR_DEVICE = 7,        /* non-finite value or fp16 overflow met on the device */
    QEVICT_ERR_CAPACITY = 8       /* a device slot pool ran out */
} qevict_status;

/* Window tiers (QEvict "Methodologie: QEvict", items 1-3). INT4 and INT8 are
 * the wider widths of the rate-distortion option ("Technische Samenvatting:
 * RDKV", 2.2); a cache allows them only with max_ledger_bits 4 or 8. */
enum { QEVICT_TIER_FP = 0, QEVICT_TIER_Q = 1, QEVICT_TIER_E = 2, QEVICT_TIER_Q4 = 3, QEVICT_TIER_Q8 = 4 };

/* Optional device-memory allocator. alloc(bytes, stream, ctx) returns a
 * device pointer (aligned to >= 256 B) or NULL; free(ptr, stream, ctx)
 * releases it. With a NULL allocator the library uses cudaMalloc/cudaFree. */
typedef struct qevict_allocator {
    void *(*alloc)(size_t bytes, void *stream, void *ctx);
    void (*free)(void *ptr, void *stream, void *ctx);
    void *ctx;
} qevict_allocator;

/* Cache geometry and budget. All sequences of the batch share one length.
 *  head_dim      must be 128; INT2 groups are 32 consecutive channels.
 *  num_q_heads   a multiple of num_kv_heads with at most 8 query heads per
 *                KV head (GQA, QEvict "Kernmechanismen", Implementatie).
 *  window        tokens per window w: a multiple of 16 in [16, 128].
 *  max_context   the longest length the cache will reach (sizes the tables).
 *  budget_frac   beta in (0, 1]: the visible tiers of each (sequence, layer)
 *                hold at most floor(beta * L * Hkv * d * 4) bytes after a
 *                routing event (QEvict, Methodologie: a budget of a few to
 *                twenty percent of the full cache).
 *  fp_share      rho in (0, 1]: the share of that budget that buys
 *                full-precision windows (the pages fix no split; 0.5 default).
 *  fp_capacity / ledger_capacity
 *                full-precision / INT2-ledger window slots per (sequence,
 *                layer); 0 derives them from the budget at max_context
 *                (plus fp_slack full-precision slots for windows that open
 *                between routing events; fp_slack 0 means 4).
 *  tier_per_kv_head
 *                0: one tier per (sequence, layer, window), shared by the KV
 *                heads. Nonzero: one tier per (sequence, KV head, layer,
 *                window) (the head-specific cache sizes of "Technische
 *                Samenvatting: DBTrimKV", Implementatie). Each (sequence, KV
 *                head) pair is then a unit with its own windows, cumulative
 *                scores (the mean mass of the head's G query heads), slot
 *                pools and budget floor(beta * L * d * 4), and its own
 *                routing. Token inputs keep their [batch][n][Hkv][head_dim]
 *                layout and q, out and mass theirs; what is per sequence in
 *                the shared mode is per unit here, unit u = b * Hkv + kvh:
 *                scores and tiers are [batch * Hkv][windows], (sequence,
 *                window) pairs name (unit, window), tier-move counts are
 *                [batch * Hkv][8], and qevict_get_view shows batch * Hkv
 *                units of 1 KV head and G query heads.
 *  max_ledger_bits
 *                0 or 2: windows are quantised to INT2 only. 4 or 8: the INT4
 *                (and INT8) tiers are allowed too ("Technische Samenvatting:
 *                RDKV", 2.2, widths {0, 2, 4, 8, 16}); ledger slots are then
 *                sized for that width. Such a cache moves windows by explicit
 *                tiers (prefill, qevict_set_tiers), listed moves and
 *                qevict_route_rd_mixed; the score, log-sparse, rate-distortion
 *                and global routes, which count INT2 bytes, reject it.
 */
typedef struct qevict_config {
    int32_t batch;
    int32_t num_layers;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t window;
    int32_t max_context;
    int32_t fp_capacity;
    int32_t ledger_capacity;
    int32_t fp_slack;
    double budget_frac;
    double fp_share;
    int32_t tier_per_kv_head;
    int32_t max_ledger_bits;
} qevict_config;

typedef struct qevict_cache qevict_cache;

/* Device layout of one layer, for inspection by tests and tools. Pointers
 * are device pointers owned by the cache; they stay valid until destroy.
 *  tier[b * max_windows + w]       uint8 tier of window w of sequence b
 *  fp_slot / ledger_slot[b*max_windows + w]
 *                                  int32 slot index or -1
 *  ledger_writes[b*max_windows+w]  int32 times window w was quantised (<= 1)
 *  fp_pool + slot * fp_slot_bytes  a full-precision window:
 *        bf16 [Hkv][2 (K, V)][2 (channels 0-63, 64-127)][window][64]
 *  ledger_pool + slot * ledger_slot_bytes   an INT2 window: [Hkv][window /
 *        16] tiles of 16 tokens, 1536 bytes each (head_dim 128):
 *        K codes at 0: [16 tokens][8] uint32, word q of a token holds
 *                 channels 16 q .. 16 q + 15, channel j at bits 2 * (j % 16);
 *        K meta at 512: [16 tokens][4 groups] half2, .x = scale, .y = min;
 *        V codes at 768: 128 uint32 words; word i = (g * 8 + mt) * 2 + h
 *                 (g, mt in 0..7, h in 0..1) holds channel 16 * mt + g + 8 h,
 *                 token t of the tile at bits 2 * t;
 *        V meta at 1280: [16 tokens][4 groups] half2.
 *        An INT4 (INT8) window keeps P = 2 (4) two-bit planes, code =
 *        sum_p 4^p c_p, each plane in the INT2 code layout; its tiles are
 *        1024 P + 512 bytes: K planes at 512 p, K meta at 512 P, V planes at
 *        512 P + 256 + 512 p, V meta at 1024 P + 256.
 *  length                          current context length (host copy). */
typedef struct qevict_view {
    int32_t batch, num_q_heads, num_kv_heads, head_dim, window;
    int32_t max_windows, num_windows;
    int32_t fp_capacity, ledger_capacity;   /* per sequence */
    int64_t length;
    int64_t fp_slot_bytes, ledger_slot_bytes;
    const uint8_t *tier;
    const int32_t *fp_slot;
    const int32_t *ledger_slot;
    const int32_t *ledger_writes;
    const uint8_t *fp_pool;
    const uint8_t *ledger_pool;
    const uint8_t *ledger_bits;   /* [b * max_windows + w] width of the ledger entry: 0, 2, 4 or 8 */
    int32_t max_ledger_bits;
    /* [b][Hkv][4] K group widths (0, 2, 4, 8) of a layer routed by
     * qevict_route_rd_kv, else NULL. Its quantised windows' ledger tiles then
     * hold, per 16 tokens: for each group in turn width / 2 planes of
     * [16 tokens][8 B] codes, the K meta [16][4] half2 (scale, minimum), the V
     * codes and V meta of the window's width; tiles at a stride of 4608 B. */
    const uint8_t *k_group_bits;
} qevict_view;

typedef struct qevict_stats {
    uint64_t demotions;       /* FP -> INT2 transitions */
    uint64_t promotions;      /* INT2 -> FP transitions */
    uint64_t evictions;       /* FP/INT2 -> evicted */
    uint64_t ledger_writes;   /* quantisations (first demotion of a window) */
    uint64_t ledger_reuses;   /* demotions that reused the ledger entry */
    int64_t device_bytes;     /* bytes the cache allocated */
} qevict_stats;

/* Host-only: the per-sequence full-precision and INT2-ledger slot counts a
 * cache created with *config gets (fp_capacity / ledger_capacity of the view)
 * and the bytes of one layer's two slot pools for the whole batch (may be
 * NULL). No routing event at any length up to max_context needs more slots:
 * full precision at most max(1, floor(rho B / c_fp)) windows (plus
 * fp_slack + 1 for windows opened between routing events and the one kept in
 * reserve for the next window), the ledger at most
 * floor(B (1 - rho) / c_q + rho B / c_fp + c_fp / c_q - 1) + 1, with B the
 * budget at max_context. INVALID_ARG for an unsupported config. */
qevict_status qevict_pool_capacity(const qevict_config *config, int32_t *fp_capacity,
                                   int32_t *ledger_capacity, int64_t *pool_bytes_per_layer);

/* Create a cache: allocates every layer's slot pools, tables and decode
 * scratch through `allocator` (NULL = cudaMalloc) on the current device and
 * initialises them on `stream`; synchronises `stream`. *out receives the
 * handle. INVALID_ARG for an unsupported geometry, OUT_OF_MEMORY when an
 * allocation fails (nothing leaks). */
qevict_status qevict_cache_create(const qevict_config *config, const qevict_allocator *allocator,
                                  void *stream, qevict_cache **out);

/* Synchronise the stream the cache was created on and release everything. */
qevict_status qevict_cache_destroy(qevict_cache *cache);

/* Fill an empty layer with n_tokens tokens and set its first tiers.
 * Semantically: append all tokens as full-precision windows, then either
 * route on `scores` ([batch][ceil(n/window)] fp32, the initial cumulative
 * window scores) or move to the tiers `tiers` ([batch][ceil(n/window)]
 * uint8). Exactly one of scores / tiers is non-NULL. Windows that end up
 * INT2 are quantised straight from k / v (their one ledger write); evicted
 * windows are never stored, so the layer never holds more than its pools.
 * k, v: bf16 [batch][n_tokens][Hkv][head_dim], read-only, caller-owned.
 * STATE if the layer is not empty; BUDGET if routing cannot hold the open
 * window. */
qevict_status qevict_prefill(qevict_cache *cache, int32_t layer, const void *k, const void *v,
                             int32_t n_tokens, const float *scores, const uint8_t *tiers,
                             void *stream);

/* Append n_new tokens to every sequence of a layer (QEvict
 * "Kernmechanismen", window-level partitioning). Token at position p goes to
 * window p / window, row p % window; a window opens in the full-precision
 * tier when its first token arrives (a slot comes from the device free
 * list; CAPACITY on the device if none is left).
 * k, v: bf16 [batch][n_new][Hkv][head_dim], caller-owned.
 * INVALID_ARG if the context would pass max_context. */
qevict_status qevict_append_kv(qevict_cache *cache, int32_t layer, const void *k, const void *v,
                               int32_t n_new, void *stream);

/* One decode step of single-token GQA attention over the tiered cache of a
 * layer, with the per-window mass that drives cumulative scoring.
 *  q     bf16 [batch][Hq][head_dim]; query head h reads KV head
 *        h / (Hq / Hkv).
 *  out   fp32 [batch][Hq][head_dim]: softmax(q K^T / sqrt(d)) V over the
 *        retained tokens. Full-precision windows are read as stored, INT2
 *        windows as min + code * scale (fp32 fma, not rounded to bf16),
 *        evicted windows are skipped and are not in the softmax denominator.
 *  mass  fp32 [batch][Hq][ceil(length/window)] or NULL: probability mass
 *        each head puts on each window (0 for evicted windows).
 *  accumulate_scores  nonzero: every window's cumulative score grows by the
 *        mean of its mass over the Hq query heads (QEvict "Cumulatieve
 *        Scoring"; RDKV 2.1 defines a token's importance as the attention it
 *        receives summed over queries).
 * INVALID_ARG for an empty layer. */
qevict_status qevict_decode_attention(qevict_cache *cache, int32_t layer, const void *q,
                                      float *out, float *mass, int32_t accumulate_scores,
                                      void *stream);

/* One decode step with this step's token fused in: equivalent to
 * qevict_append_kv(layer, k_new, v_new, n_new = 1) followed by
 * qevict_decode_attention(layer, q, out, mass, accumulate_scores), in one
 * launch. k_new, v_new: bf16 [batch][Hkv][head_dim]. mass rows are
 * ceil((length + 1) / window) long. The attention reads the cache as it was
 * plus the new token; the token is written into its window (opening one in
 * the full-precision tier when needed) after the attention, by the last CTA
 * of each sequence. INVALID_ARG if the context would pass max_context. */
qevict_status qevict_decode_step(qevict_cache *cache, int32_t layer, const void *q, const void *k_new,
                                 const void *v_new, float *out, float *mass, int32_t accumulate_scores,
                                 void *stream);

/* A routing event for a layer (QEvict "Kernmechanismen": rank windows by
 * cumulative score and move them between tiers under the byte budget).
 * Optional inputs, [batch][ceil(length/window)] fp32 or NULL:
 *  scores_override  replaces the cumulative scores before ranking;
 *  score_mult       multiplies them (drift or decay) before ranking.
 * Rule: candidates are the non-evicted windows (eviction is permanent); the
 * last window, which appends go into, stays full precision; B = floor(beta *
 * length * Hkv * d * 4); n_fp = min(C, max(1, floor(rho * B / c_fp))),
 * n_q = min(C - n_fp, floor((B - n_fp * c_fp) / c_q)) with c_fp = window *
 * Hkv * d * 4 and c_q = window * Hkv * 2 * (d / 4 + 4 * d / 32); rank by
 * score, highest first, ties to the lower window index; the top n_fp are
 * full precision, the next n_q INT2, the rest evicted. Transitions run
 * evict -> demote -> promote. A demotion quantises only a window without a
 * ledger entry (write-once ledger); a promotion dequantises the ledger codes
 * to bf16 (bf16_rne(fmaf(code, scale, min))) and keeps the ledger entry.
 * BUDGET if B < c_fp. A non-finite score among the candidates sets the
 * device status DEVICE and leaves the tiers unchanged. */
qevict_status qevict_route(qevict_cache *cache, int32_t layer, const float *scores_override,
                           const float *score_mult, void *stream);

/* A routing event whose tier counts come from a rate-distortion allocation
 * ("Technische Samenvatting: RDKV", 2.1-2.2: minimise sum w_u 2^(-b_u) over
 * bit widths b_u under a byte budget by Lagrangian relaxation over discrete
 * widths) instead of the fp_share split. Units are windows, widths the tiers'
 * (0 evicted, 2 INT2, 16 bf16), the weight w_u the window's cumulative score
 * (the attention it has received). The open window is full precision first;
 * then upgrades E -> INT2 (removing 3/4 w_u, costing c_q bytes) and INT2 ->
 * FP (removing 1/4 - 2^-16 of w_u, costing c_fp - c_q) are taken in order of
 * distortion removed per byte, highest first (E -> INT2 first on a tie, then
 * by window rank), while the gain is positive, until the first that does not
 * fit the budget floor(beta * L * Hkv * d * 4). That fixes n_fp and n_q; the
 * windows are then assigned by score rank and moved as in qevict_route
 * (same scores_override / score_mult, same errors). The comparisons are done
 * in float64. */
qevict_status qevict_route_rd(qevict_cache *cache, int32_t layer, const float *scores_override,
                              const float *score_mult, void *stream);

/* The rate-distortion routing event over all widths the cache allows
 * ("Technische Samenvatting: RDKV", 2.1-2.2: widths {0, 2, 4, 8, 16}, the
 * Lagrangian relaxation of the multiple-choice knapsack). A window's options
 * form a chain of widths: 0, 2, 4, 8, 16 (the quantised ones up to
 * max_ledger_bits, INT2 alone when it is 0 or 2) for a window never
 * quantised, and 0, b, 16 for one whose ledger entry has width b (the
 * write-once ledger fixes the width). A window of b bits costs
 * window * Hkv * 2 * (d * b / 8 + 4 * d / 32) bytes (bf16: c_fp). The open
 * window (the first of the score rank of qevict_route) is full precision;
 * every other candidate's chain step a -> b is an upgrade whose gain per
 * byte is (2^-a - 2^-b) / (cost(b) - cost(a)) * s, s its cumulative score,
 * rounded in float64 as written. Upgrades are taken by gain, highest first (a
 * lower step, then the higher-ranked window, on a tie), while the gain is
 * positive, until the first that does not fit the budget
 * floor(beta * L * Hkv * d * 4). Each window gets the width its taken steps
 * reach and is moved as in qevict_route (a demotion quantises at that width
 * when the window has no ledger entry; a promotion dequantises the entry).
 * On a cache of INT2 only this is the allocation of qevict_route_rd. Same
 * scores_override / score_mult and errors as qevict_route; allowed at every
 * max_ledger_bits. */
qevict_status qevict_route_rd_mixed(qevict_cache *cache, int32_t layer, const float *scores_override,
                                    const float *score_mult, void *stream);

/* The distortion weights of the K-cache channels ("Technische Samenvatting:
 * RDKV", 2.1: w_c = (1/sqrt(d)) ||Q[:, c]||_2 ||K[:, c]||_2; 2.2 Fase 1: once,
 * after the prefill, from the uncompressed cache), per sequence, KV head and
 * channel. Reads nothing of the cache but its shapes.
 *  q_obs    bf16 [batch][n_q][Hq][head_dim], device, 16-byte aligned: query
 *           vectors observed over the prefill; the G query heads of a KV head
 *           pool their columns (n_q * G rows per channel).
 *  k_full   bf16 [batch][n_tokens][Hkv][head_dim], device, 16-byte aligned:
 *           the layer's keys as given to qevict_prefill.
 *  weights  fp32 [batch][Hkv][head_dim], device, written. Sums of squares in
 *           fp32 in a fixed order (eight contiguous shares of the rows, each
 *           over 32 interleaved row groups, then the shares in order), then
 *           their roots: every call gives the same weights.
 * INVALID_ARG for NULL or misaligned pointers, non-positive counts or a cache
 * with tiers per KV head. */
qevict_status qevict_k_channel_weights(qevict_cache *cache, int32_t layer, const void *q_obs, int64_t n_q,
                                      const void *k_full, int64_t n_tokens, float *weights, void *stream);

/* The rate-distortion routing event with RDKV's K-channel half ("Technische
 * Samenvatting: RDKV", 2.2 Fase 2 and 3, 2.3 Zone A). First the window widths
 * of qevict_route_rd_mixed (every window is then full precision or evicted,
 * so each has the chain 0, 2, 4, 8, 16). Then, per sequence, the 32-channel K
 * groups of all KV heads take widths {0, 2, 4, 8} within the bytes the K
 * halves of the quantised windows have at their widths: a group costs 4 b + 4
 * bytes per token (codes, and the fp16 scale and minimum it always keeps),
 * its weight W is the sum of its channels' weights (float32 from
 * qevict_k_channel_weights, added in channel order in float64), and from all
 * groups at 0 the steps a -> b of gain (2^-a - 2^-b) / (tokens * (cost(b) -
 * cost(a))) * W per byte are taken by gain, highest first (a lower step, then
 * the lower (KV head, group) on a tie), while positive, until the first that
 * does not fit. The quantised windows' K groups are quantised at those
 * widths (width 0: no codes, zero meta, the channels leave the logits), their
 * V at the window's width; decoding reads both. The widths are fixed with the
 * layer's first quantisation: the call needs a layer none of whose windows
 * has a ledger entry (STATE in the device status otherwise), and afterwards
 * the layer takes appends and decodes but no further tier moves (routes,
 * listed moves and qevict_set_tiers return STATE).
 *  weights  fp32 [batch][Hkv][head_dim], device (qevict_k_channel_weights).
 * INVALID_ARG unless the cache has max_ledger_bits 8, shared tiers and at
 * most 16 KV heads; otherwise the errors of qevict_route_rd_mixed. The
 * widths can be read through qevict_get_view (k_group_bits). */
qevict_status qevict_route_rd_kv(qevict_cache *cache, int32_t layer, const float *weights,
                                 const float *scores_override, void *stream);

/* A routing event by position instead of score ("Technische Samenvatting:
 * LogQuant", Methodologie 1-2: attention peaks thin out logarithmically with
 * the distance to the current token, so the kept positions thin out the same
 * way). Windows are ranked by age (0 = the open window): the recent_windows
 * newest are dense; before them, region l = 1, 2, ... covers ages
 * [R 2^(l-1), R 2^l) (R = recent_windows) and its windows join at spacing
 * 2^l in the first round and at half the previous spacing in each later
 * round; the rank is (round, region, age), lowest first. The budget, the
 * counts and the transitions are qevict_route's, with this rank in place of
 * the score: the first n_fp windows of the order (the open one always among
 * them) stay or become full precision, the next n_q INT2, the rest evicted.
 * The cumulative scores are neither read nor changed. INVALID_ARG if
 * recent_windows < 1, BUDGET as qevict_route. */
qevict_status qevict_route_logsparse(qevict_cache *cache, int32_t layer, int32_t recent_windows, void *stream);

/* One routing event over all layers of the cache under one byte budget per
 * sequence ("Technische Samenvatting: DBTrimKV", section 3: one global budget
 * instead of budgets per layer or head, every cached entry ranked globally
 * by one utility score; the utility here is the cumulative attention score,
 * on one scale across layers because each layer spreads one unit of mass per
 * query head per decode step). The per-layer rule of qevict_route is applied
 * with the candidates, the budget and the forced windows widened to all
 * layers (and KV heads, with per-head tiers) of a sequence:
 *   budget B = floor(beta * sum over layers and units of L * Hkv * d * 4);
 *   the last window of every unit of every layer is forced full precision;
 *   n_fp = min(C, max(forced, floor(rho * B / c_fp))),
 *   n_q = min(C - n_fp, floor((B - n_fp * c_fp) / c_q)), c_fp and c_q of one
 *   unit's window; rank by score descending, then (layer, unit, window)
 *   ascending; the top n_fp full precision, the next n_q INT2, the rest
 *   evicted, with the transitions of qevict_route in every layer.
 * Layers may end up with different numbers of windows, so a layer can need
 * more slots than its pools were sized for from its own budget share: size
 * fp_capacity and ledger_capacity for it (a layer whose pool runs out sets
 * CAPACITY and keeps its tiers).
 *  scores_override  NULL, or a HOST array of num_layers pointers, each NULL
 *                   or a device fp32 [units][ceil(length / window)] array
 *                   that replaces that layer's cumulative scores first.
 * BUDGET (host) if the forced windows alone pass the budget. A non-finite
 * score among the candidates sets DEVICE and leaves every layer's tiers
 * unchanged. Uses one table of ranking keys per cache: do not overlap two
 * global events of one cache. */
qevict_status qevict_route_global(qevict_cache *cache, const float *const *scores_override, void *stream);

/* Demote the listed windows FP -> INT2 (QEvict "Demotie"), in list order.
 * bw_ids: int32 [n][2] device array of (sequence, window) pairs. A window
 * without a ledger entry is quantised per token, KV head and group of 32
 * channels: min16 = fp16(min), scale16 = fp16(fl32(fl32(max - min) / 3)),
 * code = clamp(rint(fl32(fl32(x - min16) / scale16)), 0, 3) (all codes 0 if
 * scale16 is 0); a window with a ledger entry reuses it. An entry naming a
 * window that is not full precision, or the partially filled last window,
 * sets STATE on the device and is skipped. */
qevict_status qevict_demote_quantize(qevict_cache *cache, int32_t layer, const int32_t *bw_ids,
                                     int32_t n, void *stream);

/* Promote the listed windows INT2 -> FP (QEvict "Promotie"), in list order:
 * x = bf16_rne(fmaf(code, scale, min)) into a new full-precision slot; the
 * ledger entry is kept for later demotions. bw_ids as above; an entry naming
 * a window that is not INT2 sets STATE and is skipped. */
qevict_status qevict_promote_dequantize(qevict_cache *cache, int32_t layer, const int32_t *bw_ids,
                                        int32_t n, void *stream);

/* Move a layer's windows to explicit tiers (uint8 [batch][ceil(length /
 * window)]), with the same transition rules as a routing event but no
 * budget. E -> FP/INT2 and a change of the partially filled last window set
 * STATE on the device and leave the tiers unchanged. */
qevict_status qevict_set_tiers(qevict_cache *cache, int32_t layer, const uint8_t *tiers,
                               void *stream);

/* Write a layer's cumulative window scores, fp32 [batch][ceil(length /
 * window)], to `scores`. */
qevict_status qevict_get_scores(qevict_cache *cache, int32_t layer, float *scores, void *stream);

/* Fill *view with the device layout of a layer (host call, no stream work). */
qevict_status qevict_get_view(const qevict_cache *cache, int32_t layer, qevict_view *view);

/* Synchronise `stream` and return the sticky device status (QEVICT_OK if no
 * device error happened since the last qevict_clear_status). */
qevict_status qevict_get_status(qevict_cache *cache, void *stream);

/* Reset the sticky device status to QEVICT_OK (enqueued on `stream`). It also
 * clears the decode scratch's split records and counters (a decode that gave
 * up waiting, QEVICT_ERR_TIMEOUT, can leave them inconsistent), so it must not
 * overlap a decode of this cache on another stream. */
qevict_status qevict_clear_status(qevict_cache *cache, void *stream);

/* Synchronise `stream` and copy the transition counters to *stats (host). */
qevict_status qevict_get_stats(qevict_cache *cache, qevict_stats *stats, void *stream);

/* Diagnostics of a layer's last completed tier move (QEvict "Kernbijdragen":
 * selection churn and latent importance reactivation, reading the
 * full-precision tier as the active set). A tier move is a routing event, a
 * prefill with scores or tiers, qevict_set_tiers, qevict_demote_quantize or
 * qevict_promote_dequantize; appends and decodes are not. Synchronises
 * `stream`, then writes int32 [batch][8] to the HOST array `counts`, per
 * sequence:
 *   [0] full-precision windows before the move   [1] INT2 windows before
 *   [2] full-precision windows after             [3] INT2 windows after
 *   [4] kept: full precision before and after    [5] promoted: INT2 -> FP
 *   [6] demoted: FP -> INT2                      [7] evicted: FP or INT2 -> E
 * Selection churn = 1 - [4] / [2]; reactivation rate = [5] / [1]. All zero
 * before the layer's first move. A move that stops on a device error (BUDGET,
 * STATE, DEVICE) leaves the previous counts. */
qevict_status qevict_get_tier_move_counts(qevict_cache *cache, int32_t layer, int32_t *counts, void *stream);

/* Future missed mass (QEvict "Kernbijdragen"): for each sequence and query
 * head, the share of softmax(q K_full^T / sqrt(d)) over all of the layer's
 * tokens that falls on tokens whose window is evicted now. A measurement, not
 * part of decoding: the caller keeps the layer's full keys, as they were
 * stored before any tier move.
 *  q       bf16 [batch][Hq][head_dim], device, 16-byte aligned.
 *  k_full  bf16 [batch][n_tokens][Hkv][head_dim], device, 16-byte aligned;
 *          n_tokens must equal the layer's length (INVALID_ARG otherwise).
 *  fmm     fp32 [batch][Hq], device; 0 where nothing is evicted.
 * Logits and sums are fp32. The call uses the cache's decode scratch, so it
 * must not overlap a decode of the same cache on another stream. */
qevict_status qevict_future_missed_mass(qevict_cache *cache, int32_t layer, const void *q, const void *k_full,
                                        int64_t n_tokens, float *fmm, void *stream);

/* Let a decode launch overlap the end of the kernel before it in the stream
 * (programmatic dependent launch): the decode kernel starts loading this
 * layer's cache while the previous kernel finishes, and waits for that kernel
 * before it reads q, k_new and v_new. The library enables it only for a
 * decode whose previous call on this cache was on another layer and on the
 * same stream. Enable it only if the operation just before each such decode
 * in the stream is a kernel (for example a graph of consecutive decode steps,
 * or the projection that produces q): a copy or memset directly before the
 * launch is not waited for. Off by default. */
qevict_status qevict_set_launch_overlap(qevict_cache *cache, int32_t enable);

/* Launch the decode grid cooperatively (enable != 0, the default) or not. The
 * splits of a (sequence, KV head) wait for one another, so all CTAs of a
 * decode must be resident together: a cooperative grid starts only when they
 * can be, so a kernel on another stream holding SMs delays the decode instead
 * of leaving its resident splits waiting for the others (up to the wait
 * limit below, then QEVICT_ERR_TIMEOUT). A cooperative grid cannot start its
 * CTAs one by one as the kernel before it frees SMs, which costs about a
 * microsecond per launch; disable it only where nothing else runs on the GPU
 * while decodes run. */
qevict_status qevict_set_cooperative_launch(qevict_cache *cache, int32_t enable);

/* Limit, in SM clock cycles (clock64), of every wait of a decode on other CTAs
 * of the same launch: the splits of a (sequence, KV head) waiting for one
 * another's records, and the wait before the fused append moves the tables.
 * A wait that runs out sets QEVICT_ERR_TIMEOUT in the status word and the
 * kernel finishes without waiting further (its outputs are then not valid);
 * waits on the CTA's own copies keep their own limit. cycles <= 0 restores the
 * default, 4e9 cycles (about two seconds at GB300 clocks). With a cooperative
 * launch all CTAs are resident together and a wait only outlasts the work of
 * the slowest split when something is wrong; a short limit is a diagnostic,
 * for tests of the timeout path. */
qevict_status qevict_set_wait_limit(qevict_cache *cache, int64_t cycles);

/* The kernels keep each layer's context length in device memory and read it
 * when they run, so a CUDA graph captured from these calls can be replayed:
 * every replay appends, attends and routes at the device-side length of the
 * moment. The host keeps a copy of each length for argument checks and
 * output shapes (mass and score rows are ceil(length / window) long at the
 * time the kernel runs). After replaying graphs, call qevict_refresh_lengths
 * (synchronises `stream`) to copy the device lengths back to the host. */
qevict_status qevict_refresh_lengths(qevict_cache *cache, void *stream);

/* Current context length of a layer (host copy), or -1 for a bad layer. */
int64_t qevict_length(const qevict_cache *cache, int32_t layer);

/* Bytes of device scratch that qevict_decode_attention_static_scratch can
 * use: 4 MiB, one array per device, owned by the library. */
#define QEVICT_STATIC_SCRATCH_BYTES (4u * 1024u * 1024u)

/* qevict_decode_attention with the kernel's per-call scratch taken from a
 * fixed 4 MiB device array that the library holds, instead of the scratch
 * block the cache drew from its allocator. The call allocates nothing: no
 * cudaMalloc, no allocator callback, no library routine that allocates.
 * The QEvict pages have no counterpart of this call; it exists for callers
 * that cannot reach an allocator when they decode, for example an engine
 * that has handed all free device memory to its own pools after set-up, or
 * a host thread that must not block on an allocator's lock.
 *
 * Arguments, outputs and errors are those of qevict_decode_attention.
 * The scratch a call needs is, per (sequence, KV head): 1 KiB per query head
 * for each decode split (up to 32 splits, as many as fit the GPU in one
 * wave), 4 KiB of split records, 8 B of counters, and 8 B per query head for
 * each 16-token tile of every slot of the cache's full-precision and ledger
 * pools (the per-claim records). A cache whose need passes
 * QEVICT_STATIC_SCRATCH_BYTES is rejected with INVALID_ARG before anything
 * is enqueued, and the error text gives both sizes. The cache's device must
 * be current (INVALID_ARG otherwise).
 *
 * Set-up: the first call on a device, with that device current, looks up the
 * array's address and clears it. That first call synchronises the device, so
 * make it before any stream capture begins. Where the counters, split
 * records and partials lie in the array depends on the cache's shape, so
 * every call clears that part of the array on `stream` before its launch
 * (cudaMemsetAsync, which allocates nothing); calls on caches of different
 * shapes can therefore follow one another on a stream.
 *
 * One array serves every cache and stream on a device: calls whose kernels
 * can overlap (other streams, other host threads, other caches) race on it
 * and give wrong results. Order them on one stream or by events. */
qevict_status qevict_decode_attention_static_scratch(qevict_cache *cache, int32_t layer, const void *q,
                                                     float *out, float *mass, int32_t accumulate_scores,
                                                     void *stream);

/* Thread-local text of the last host-side error of this thread. */
const char *qevict_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* QEVICT_H */
