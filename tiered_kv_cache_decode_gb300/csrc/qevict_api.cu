// Host side of the C ABI declared in include/qevict.h: configuration checks,
// slot-pool sizing from the byte budget, device allocations, host-side error
// reporting and the launch sequence of every call.
#include "qevict_internal.cuh"

#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <mutex>
#include <string>
#include <vector>

using namespace qevict;

namespace {

thread_local std::string g_last_error;

qevict_status fail(qevict_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

qevict_status cuda_fail(cudaError_t e, const char *what) {
    return fail(QEVICT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct LayerHost {
    LayerDev dev{};
    bool kch = false;       // routed by qevict_route_rd_kv: no further tier moves
    CUtensorMap tmap{};     // 4-D tiled view of the full-precision pool, 64 x 16 x 4 boxes
    int64_t length = 0;
    void *base = nullptr;
};

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

}  // namespace

struct qevict_cache {
    qevict_config cfg{};
    qevict_allocator alloc{};
    bool user_alloc = false;
    cudaStream_t stream = nullptr;
    int device = 0;
    int num_sms = 1;
    int Wmax = 0, CF = 0, CQ = 0, G = 0;
    int64_t c_fp = 0, c_q = 0;
    std::vector<LayerHost> layers;
    CacheDev cdev{};
    DecodeScratch scratch{};
    void *cbase = nullptr;
    int64_t total_bytes = 0;
    std::vector<void *> blocks;
    // the last operation enqueued: programmatic dependent launch is used for a
    // decode only when that operation was on another layer and on the same stream
    int prev_layer = -1;
    void *prev_stream = nullptr;
    void *scratch_base = nullptr;
    size_t scratch_bytes = 0;
    // global routing: the layers' device descriptors, ranking keys, thresholds, flags
    int hs = 1;   // KV heads folded into each unit (per-head tiers), else 1
    void *groute_base = nullptr;
    size_t groute_bytes = 0;
    LayerDev *ldev = nullptr;
    unsigned long long *gkeys = nullptr, *gthr = nullptr;
    int32_t *gflag = nullptr, *gcnt = nullptr;
    bool allow_pdl = false;    // qevict_set_launch_overlap
    bool coop = true;          // qevict_set_cooperative_launch
};

namespace {

void *dev_alloc(qevict_cache *c, size_t bytes) {
    void *p = nullptr;
    if (c->user_alloc) {
        p = c->alloc.alloc(bytes, (void *)c->stream, c->alloc.ctx);
    } else if (cudaMalloc(&p, bytes) != cudaSuccess) {
        cudaGetLastError();
        p = nullptr;
    }
    if (p) {
        c->blocks.push_back(p);
        c->total_bytes += (int64_t)bytes;
    }
    return p;
}

void release_all(qevict_cache *c) {
    for (void *p : c->blocks) {
        if (c->user_alloc) c->alloc.free(p, (void *)c->stream, c->alloc.ctx);
        else cudaFree(p);
    }
    c->blocks.clear();
}

struct Carver {
    size_t off = 0;
    size_t take(size_t bytes) {
        const size_t o = off;
        off += (bytes + 255) & ~size_t(255);
        return o;
    }
};

// Window costs per sequence: full-precision K+V bf16, INT2 codes + fp16 meta.
void window_costs(int w, int Hkv, int64_t *c_fp, int64_t *c_q) {
    *c_fp = (int64_t)w * Hkv * kHeadDim * 4;
    *c_q = (int64_t)w * Hkv * 2 * (kHeadDim / 4 + 4 * (kHeadDim / kGroup));
}

int64_t budget_bytes(const qevict_config &cfg, int64_t L) {
    const int64_t F = L * cfg.num_kv_heads * kHeadDim * 4;
    return (int64_t)floor(cfg.budget_frac * (double)F);
}

int fp_budget_windows(int64_t Bt, int64_t c_fp, double rho) {  // host copy of the plan kernel's rule
    return (int)floor((rho * (double)Bt) / (double)c_fp);
}

qevict_status check_layer(const qevict_cache *c, int32_t layer) {
    if (!c) return fail(QEVICT_ERR_INVALID_ARG, "cache is NULL");
    if (layer < 0 || layer >= c->cfg.num_layers)
        return fail(QEVICT_ERR_INVALID_ARG, "layer %d out of range [0, %d)", layer, c->cfg.num_layers);
    return QEVICT_OK;
}

int n_windows(const qevict_cache *c, int64_t L) { return (int)((L + c->cfg.window - 1) / c->cfg.window); }

// The score, log-sparse, rate-distortion and global routes count INT2 bytes for
// every quantised window, so a cache that allows wider widths does not take them.
qevict_status check_int2_only(const qevict_cache *c, const char *what) {
    if (c->cfg.max_ledger_bits > 2)
        return fail(QEVICT_ERR_INVALID_ARG, "%s counts INT2 bytes; this cache allows %d-bit windows "
                    "(route it with qevict_route_rd_mixed or explicit tiers)", what, c->cfg.max_ledger_bits);
    return QEVICT_OK;
}

void note_op(qevict_cache *c, int layer, void *stream) {
    c->prev_layer = layer;
    c->prev_stream = stream;
}

// Plan + the data movement it queues, in order: quantise (reads full-precision
// slots released by demotions), then promote / prefill copy (write slots).
qevict_status run_plan(qevict_cache *c, LayerHost &lh, const PlanArgs &a, const __nv_bfloat16 *k_ext,
                       const __nv_bfloat16 *v_ext, cudaStream_t s) {
    if (lh.kch && a.mode != PLAN_RD_KV)
        return fail(QEVICT_ERR_STATE, "layer %d has K-channel widths and takes no further tier moves", a.layer);
    cudaError_t e = launch_plan(lh.dev, c->cdev, a, s);
    if (e != cudaSuccess) return cuda_fail(e, "plan kernel");
    const int maxf = c->Wmax < c->CF ? c->Wmax : c->CF;
    const bool prefill = a.mode == PLAN_PREFILL_SCORES || a.mode == PLAN_PREFILL_TIERS;
    // a plan quantises at most the windows it demotes from full precision (or, in a
    // prefill, every window): the grids are sized for that many entries
    int maxq = c->Wmax < c->CQ ? c->Wmax : c->CQ;
    if (!prefill && maxf < maxq) maxq = maxf;
    if (a.mode != PLAN_PROMOTE) {
        e = launch_quantize(lh.dev, c->cdev, a.layer, k_ext, v_ext, a.prefill_len, maxq, s);
        if (e != cudaSuccess) return cuda_fail(e, "quantize kernel");
    }
    if (prefill) {
        e = launch_prefill_copy(lh.dev, k_ext, v_ext, a.prefill_len, maxf, s);
        if (e != cudaSuccess) return cuda_fail(e, "prefill copy kernel");
    } else if (a.mode != PLAN_DEMOTE) {
        e = launch_promote(lh.dev, c->cdev, maxf, s);
        if (e != cudaSuccess) return cuda_fail(e, "promote kernel");
    }
    note_op(c, a.layer, (void *)s);
    return QEVICT_OK;
}

// Pool sizes that no routing event up to max_context can exceed. The budget
// grows with the length, so the full-precision count peaks at max_context;
// n_fp + n_q does not (it drops when n_fp steps up), so the ledger uses the
// bound n_fp + n_q <= B (1 - rho) / c_q + rho B / c_fp + c_fp / c_q - 1, which
// follows from n_fp c_fp + n_q c_q <= B and n_fp >= rho B / c_fp - 1 and
// increases with B.
void pool_capacity(const qevict_config &cfg, int Wmax, int64_t c_fp, int64_t c_q, int *CF, int *CQ) {
    const int64_t Bmax = budget_bytes(cfg, cfg.max_context);
    int nfp = fp_budget_windows(Bmax, c_fp, cfg.fp_share);
    if (nfp < 1) nfp = 1;
    if (nfp > Wmax) nfp = Wmax;
    const double rho = cfg.fp_share, Bd = (double)Bmax;
    const double lq = Bd * (1.0 - rho) / (double)c_q + rho * Bd / (double)c_fp + (double)c_fp / (double)c_q - 1.0;
    int64_t nl = (int64_t)floor(lq) + 1;
    if (nl > Wmax) nl = Wmax;
    if (nl < 1) nl = 1;
    const int slack = cfg.fp_slack > 0 ? cfg.fp_slack : 4;
    *CF = cfg.fp_capacity > 0 ? cfg.fp_capacity : (nfp + slack + 1 < Wmax ? nfp + slack + 1 : Wmax);
    *CQ = cfg.ledger_capacity > 0 ? cfg.ledger_capacity : (int)nl;
}

qevict_status check_config(const qevict_config &cfg) {
    if (cfg.batch < 1 || cfg.num_layers < 1 || cfg.num_kv_heads < 1 || cfg.num_q_heads < 1)
        return fail(QEVICT_ERR_INVALID_ARG, "batch, layers and head counts must be >= 1");
    if (cfg.num_q_heads % cfg.num_kv_heads != 0 || cfg.num_q_heads / cfg.num_kv_heads > kMaxG)
        return fail(QEVICT_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads, at most %d per KV head",
                    kMaxG);
    if (cfg.head_dim != kHeadDim) return fail(QEVICT_ERR_INVALID_ARG, "head_dim must be %d", kHeadDim);
    if (cfg.max_ledger_bits != 0 && cfg.max_ledger_bits != 2 && cfg.max_ledger_bits != 4 && cfg.max_ledger_bits != 8)
        return fail(QEVICT_ERR_INVALID_ARG, "max_ledger_bits must be 0, 2, 4 or 8");
    if (cfg.window < 16 || cfg.window > 128 || cfg.window % kVTile != 0)
        return fail(QEVICT_ERR_INVALID_ARG, "window must be a multiple of 16 in [16, 128]");
    if (cfg.max_context < 1) return fail(QEVICT_ERR_INVALID_ARG, "max_context must be >= 1");
    if (!(cfg.budget_frac > 0.0 && cfg.budget_frac <= 1.0))
        return fail(QEVICT_ERR_INVALID_ARG, "budget_frac must be in (0, 1]");
    if (!(cfg.fp_share > 0.0 && cfg.fp_share <= 1.0))
        return fail(QEVICT_ERR_INVALID_ARG, "fp_share must be in (0, 1]");
    if (cfg.fp_capacity < 0 || cfg.ledger_capacity < 0 || cfg.fp_slack < 0)
        return fail(QEVICT_ERR_INVALID_ARG, "capacities must be >= 0");
    const int Wmax = (cfg.max_context + cfg.window - 1) / cfg.window;
    if (Wmax > 4096) return fail(QEVICT_ERR_INVALID_ARG, "at most 4096 windows per sequence (got %d)", Wmax);
    if ((int64_t)cfg.num_layers * (cfg.tier_per_kv_head ? cfg.num_kv_heads : 1) * Wmax > 0xffffffffll)
        return fail(QEVICT_ERR_INVALID_ARG, "layers x windows (x KV heads with per-head tiers) must be below 2^32");
    if (cfg.tier_per_kv_head && (int64_t)cfg.batch * cfg.num_kv_heads > 65535)
        return fail(QEVICT_ERR_INVALID_ARG, "with per-head tiers batch x num_kv_heads must be at most 65535");
    return QEVICT_OK;
}

// The configuration the cache works with: with per-head tiers every
// (sequence, KV head) pair is a unit of 1 KV head and G query heads.
qevict_config unit_config(const qevict_config &cfg) {
    qevict_config u = cfg;
    if (cfg.tier_per_kv_head) {
        u.batch = cfg.batch * cfg.num_kv_heads;
        u.num_q_heads = cfg.num_q_heads / cfg.num_kv_heads;
        u.num_kv_heads = 1;
    }
    return u;
}

}  // namespace

extern "C" {

qevict_status qevict_pool_capacity(const qevict_config *config, int32_t *fp_capacity, int32_t *ledger_capacity,
                                   int64_t *pool_bytes_per_layer) {
    if (!config || !fp_capacity || !ledger_capacity) return fail(QEVICT_ERR_INVALID_ARG, "NULL argument");
    qevict_status st = check_config(*config);
    if (st) return st;
    const qevict_config cfg = unit_config(*config);
    const int Wmax = (cfg.max_context + cfg.window - 1) / cfg.window;
    int64_t c_fp, c_q;
    window_costs(cfg.window, cfg.num_kv_heads, &c_fp, &c_q);
    int CF, CQ;
    pool_capacity(cfg, Wmax, c_fp, c_q, &CF, &CQ);
    *fp_capacity = CF;
    *ledger_capacity = CQ;
    if (pool_bytes_per_layer) {
        const int maxP = cfg.max_ledger_bits > 2 ? cfg.max_ledger_bits / 2 : 1;
        const int64_t lgs = (int64_t)cfg.num_kv_heads * (cfg.window / 16) * qtile_bytes(maxP);
        *pool_bytes_per_layer = (int64_t)cfg.batch * (CF * c_fp + CQ * lgs);
    }
    return QEVICT_OK;
}

const char *qevict_last_error(void) { return g_last_error.c_str(); }

qevict_status qevict_cache_create(const qevict_config *config, const qevict_allocator *allocator, void *stream,
                                  qevict_cache **out) {
    if (!config || !out) return fail(QEVICT_ERR_INVALID_ARG, "config and out must not be NULL");
    *out = nullptr;
    {
        const qevict_status cs = check_config(*config);
        if (cs) return cs;
    }
    const qevict_config cfg = unit_config(*config);
    const int hs = config->tier_per_kv_head ? config->num_kv_heads : 1;
    const int Wmax = (cfg.max_context + cfg.window - 1) / cfg.window;
    if (allocator && (!allocator->alloc || !allocator->free))
        return fail(QEVICT_ERR_INVALID_ARG, "allocator needs both alloc and free");

    qevict_cache *c = new qevict_cache();
    c->cfg = cfg;
    if (allocator) {
        c->alloc = *allocator;
        c->user_alloc = true;
    }
    c->stream = (cudaStream_t)stream;
    cudaGetDevice(&c->device);
    cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
    c->G = cfg.num_q_heads / cfg.num_kv_heads;
    c->Wmax = Wmax;
    window_costs(cfg.window, cfg.num_kv_heads, &c->c_fp, &c->c_q);
    pool_capacity(cfg, Wmax, c->c_fp, c->c_q, &c->CF, &c->CQ);
    const int B = cfg.batch, Hkv = cfg.num_kv_heads, Hq = cfg.num_q_heads, w = cfg.window;
    const int64_t fps = (int64_t)Hkv * 2 * w * kHeadDim * 2;
    const int maxP = cfg.max_ledger_bits > 2 ? cfg.max_ledger_bits / 2 : 1;
    const int64_t lgs = (int64_t)Hkv * (w / 16) * qtile_bytes(maxP);   // ledger slots sized for the widest width

    cudaError_t err = cudaSuccess;
    // cache-wide status and statistics
    c->cbase = dev_alloc(c, 256);
    if (!c->cbase) {
        release_all(c);
        delete c;
        return fail(QEVICT_ERR_OUT_OF_MEMORY, "allocation of 256 B failed");
    }
    c->cdev.status = reinterpret_cast<int32_t *>(c->cbase);
    c->cdev.stats = reinterpret_cast<unsigned long long *>((uint8_t *)c->cbase + 64);
    c->cdev.wait_cycles = kDefaultWaitCycles;

    // every allocation first, so that a failing allocator leaves nothing behind
    {
        Carver cv;
        const int rec_stride = decode_records(c->CF, c->CQ, cfg.window, maxP);
        const size_t o_part = cv.take((size_t)B * Hkv * kMaxSplits * c->G * kHeadDim * 8);
        const size_t o_stat = cv.take((size_t)B * Hkv * kMaxSplits * kMaxG * 16);
        const size_t o_rec = cv.take((size_t)B * Hkv * rec_stride * c->G * 8);
        // the future-missed-mass partials (12 B per split and query head)
        const size_t o_ws = cv.take((size_t)B * Hq * (Wmax * 8 > 12 ? Wmax * 8 : 12));
        const size_t o_bar = cv.take((size_t)B * Hkv * 8);
        const size_t o_ab = cv.take((size_t)B * 4);
        uint8_t *base = (uint8_t *)dev_alloc(c, cv.off);
        if (!base) {
            const size_t need = cv.off;
            release_all(c);
            delete c;
            return fail(QEVICT_ERR_OUT_OF_MEMORY, "allocation of %zu B of decode scratch failed", need);
        }
        c->scratch.part = (unsigned long long *)(base + o_part);
        c->scratch.stat = (unsigned long long *)(base + o_stat);
        c->scratch.rec = (float2 *)(base + o_rec);
        c->scratch.rec_stride = rec_stride;
        c->scratch.wstat = (float2 *)(base + o_ws);
        c->scratch.bar = (uint32_t *)(base + o_bar);
        c->scratch.arrive_b = (uint32_t *)(base + o_ab);
        c->scratch_bytes = cv.off;
        c->scratch_base = base;
    }
    c->hs = hs;
    {
        const int S = B / hs;
        Carver cv;
        const size_t o_ld = cv.take((size_t)cfg.num_layers * sizeof(LayerDev));
        const size_t o_gk = cv.take((size_t)S * cfg.num_layers * hs * Wmax * 8);
        const size_t o_gt = cv.take((size_t)S * 16);
        const size_t o_gf = cv.take((size_t)S * 4);
        const size_t o_gc = cv.take((size_t)S * 16);
        uint8_t *base = (uint8_t *)dev_alloc(c, cv.off);
        if (!base) {
            const size_t need = cv.off;
            release_all(c);
            delete c;
            return fail(QEVICT_ERR_OUT_OF_MEMORY, "allocation of %zu B of routing tables failed", need);
        }
        c->ldev = (LayerDev *)(base + o_ld);
        c->gkeys = (unsigned long long *)(base + o_gk);
        c->gthr = (unsigned long long *)(base + o_gt);
        c->gflag = (int32_t *)(base + o_gf);
        c->gcnt = (int32_t *)(base + o_gc);
        c->groute_base = base;
        c->groute_bytes = cv.off;
    }
    c->layers.resize(cfg.num_layers);
    for (int l = 0; l < cfg.num_layers; ++l) {
        LayerDev &D = c->layers[l].dev;
        D.B = B;
        D.hs = hs;
        D.maxP = maxP;
        D.Hq = Hq;
        D.Hkv = Hkv;
        D.G = c->G;
        D.w = w;
        D.Wmax = Wmax;
        D.CF = c->CF;
        D.CQ = c->CQ;
        D.max_context = cfg.max_context;
        D.beta = cfg.budget_frac;
        D.rho = cfg.fp_share;
        D.c_fp = c->c_fp;
        D.c_q = c->c_q;
        D.fp_slot_bytes = fps;
        D.lg_slot_bytes = lgs;
        Carver cv;
        const size_t o_fp = cv.take((size_t)B * c->CF * fps);
        const size_t o_lg = cv.take((size_t)B * c->CQ * lgs);
        const size_t o_tier = cv.take((size_t)B * Wmax);
        const size_t o_fps = cv.take((size_t)B * Wmax * 4);
        const size_t o_lgs = cv.take((size_t)B * Wmax * 4);
        const size_t o_lw = cv.take((size_t)B * Wmax * 4);
        const size_t o_sc = cv.take((size_t)B * Hkv * Wmax * 4);
        const size_t o_ff = cv.take((size_t)B * c->CF * 4);
        const size_t o_lf = cv.take((size_t)B * c->CQ * 4);
        const size_t o_fl = cv.take((size_t)B * c->CF * 8);
        const size_t o_ql = cv.take((size_t)B * c->CQ * 8);
        const size_t o_ctr = cv.take((size_t)B * kCtrN * 4);
        const size_t o_wq = cv.take((size_t)B * Wmax * 16);
        const size_t o_wp = cv.take((size_t)B * Wmax * 16);
        const size_t o_wc = cv.take((size_t)B * Wmax * 16);
        const size_t o_dg = cv.take((size_t)B * 8 * 4);
        const size_t o_lb = cv.take((size_t)B * Wmax);
        const size_t o_kg = cv.take((size_t)B * Hkv * kGroups);
        uint8_t *base = (uint8_t *)dev_alloc(c, cv.off);
        if (!base) {
            const size_t need = cv.off;
            release_all(c);
            delete c;
            return fail(QEVICT_ERR_OUT_OF_MEMORY, "allocation of %zu B for layer %d failed", need, l);
        }
        c->layers[l].base = base;
        D.fp_pool = base + o_fp;
        D.lg_pool = base + o_lg;
        D.tier = base + o_tier;
        D.fp_slot = (int32_t *)(base + o_fps);
        D.lg_slot = (int32_t *)(base + o_lgs);
        D.lwrites = (int32_t *)(base + o_lw);
        D.score_part = (float *)(base + o_sc);
        D.fp_free = (int32_t *)(base + o_ff);
        D.lg_free = (int32_t *)(base + o_lf);
        D.fp_list = (int2 *)(base + o_fl);
        D.q_list = (int2 *)(base + o_ql);
        D.ctr = (int32_t *)(base + o_ctr);
        D.work_q = (int4 *)(base + o_wq);
        D.work_p = (int4 *)(base + o_wp);
        D.work_c = (int4 *)(base + o_wc);
        D.diag = (int32_t *)(base + o_dg);
        D.lbits = base + o_lb;
        D.kgw = base + o_kg;
    }
    err = prepare_decode();
    EncodeTiledFn enc = encode_tiled();
    for (int l = 0; l < cfg.num_layers && err == cudaSuccess; ++l) {
        if (!enc) {
            err = cudaErrorNotSupported;
            break;
        }
        // the full-precision pool as [slot * Hkv + kvh][K0, K1, V0, V1][token][64 channels]
        const LayerDev &D = c->layers[l].dev;
        const cuuint64_t dims[4] = {64, (cuuint64_t)w, 4, (cuuint64_t)B * c->CF * Hkv};
        const cuuint64_t strides[3] = {128, (cuuint64_t)w * 128, (cuuint64_t)w * 512};
        const cuuint32_t box[4] = {64, 16, 4, 1};   // the K and V of a 16-token unit
        const cuuint32_t estr[4] = {1, 1, 1, 1};
        CUresult r = enc(&c->layers[l].tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, D.fp_pool, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) err = cudaErrorInvalidValue;
    }
    if (err == cudaSuccess) err = cudaMemsetAsync(c->cbase, 0, 256, c->stream);
    if (err == cudaSuccess) err = cudaMemsetAsync(c->scratch_base, 0, c->scratch_bytes, c->stream);
    if (err == cudaSuccess) err = cudaMemsetAsync(c->groute_base, 0, c->groute_bytes, c->stream);
    std::vector<LayerDev> ltab(cfg.num_layers);   // alive until the synchronisation below
    for (int l = 0; l < cfg.num_layers; ++l) ltab[l] = c->layers[l].dev;
    if (err == cudaSuccess)
        err = cudaMemcpyAsync(c->ldev, ltab.data(), ltab.size() * sizeof(LayerDev), cudaMemcpyHostToDevice,
                              c->stream);
    for (int l = 0; l < cfg.num_layers && err == cudaSuccess; ++l) {
        err = launch_init_layer(c->layers[l].dev, c->stream);
        if (err == cudaSuccess) err = cudaMemsetAsync(c->layers[l].dev.diag, 0, (size_t)B * 8 * 4, c->stream);
    }
    if (err == cudaSuccess) err = cudaStreamSynchronize(c->stream);
    if (err != cudaSuccess) {
        release_all(c);
        delete c;
        return cuda_fail(err, "cache initialisation");
    }
    *out = c;
    return QEVICT_OK;
}

qevict_status qevict_cache_destroy(qevict_cache *cache) {
    if (!cache) return fail(QEVICT_ERR_INVALID_ARG, "cache is NULL");
    cudaStreamSynchronize(cache->stream);
    release_all(cache);
    delete cache;
    return QEVICT_OK;
}

qevict_status qevict_prefill(qevict_cache *c, int32_t layer, const void *k, const void *v, int32_t n_tokens,
                             const float *scores, const uint8_t *tiers, void *stream) {
    qevict_status st = check_layer(c, layer);
    if (st) return st;
    LayerHost &lh = c->layers[layer];
    if (!k || !v) return fail(QEVICT_ERR_INVALID_ARG, "k and v must not be NULL");
    if ((scores == nullptr) == (tiers == nullptr))
        return fail(QEVICT_ERR_INVALID_ARG, "give exactly one of scores and tiers");
    if (scores) {
        const qevict_status cs = check_int2_only(c, "a prefill with scores");
        if (cs) return cs;
    }
    if (n_tokens < 1 || n_tokens > c->cfg.max_context)
        return fail(QEVICT_ERR_INVALID_ARG, "n_tokens %d out of [1, %d]", n_tokens, c->cfg.max_context);
    if (lh.length != 0) return fail(QEVICT_ERR_STATE, "prefill needs an empty layer (length %lld)", (long long)lh.length);
    PlanArgs a{};
    a.mode = scores ? PLAN_PREFILL_SCORES : PLAN_PREFILL_TIERS;
    a.layer = layer;
    a.prefill_len = n_tokens;
    a.scores = scores;
    a.tiers = tiers;
    if (scores) {
        const int64_t Bt = budget_bytes(c->cfg, n_tokens);
        if (Bt < c->c_fp)
            return fail(QEVICT_ERR_BUDGET, "budget %lld B cannot hold the open window (%lld B)", (long long)Bt,
                        (long long)c->c_fp);
    }
    st = run_plan(c, lh, a, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, (cudaStream_t)stream);
    if (st) return st;
    lh.length = n_tokens;
    return QEVICT_OK;
}

qevict_status qevict_append_kv(qevict_cache *c, int32_t layer, const void *k, const void *v, int32_t n_new,
                               void *stream) {
    qevict_status st = check_layer(c, layer);
    if (st) return st;
    LayerHost &lh = c->layers[layer];
    if (!k || !v) return fail(QEVICT_ERR_INVALID_ARG, "k and v must not be NULL");
    if (n_new < 1) return fail(QEVICT_ERR_INVALID_ARG, "n_new must be >= 1");
    if (lh.length + n_new > c->cfg.max_context)
        return fail(QEVICT_ERR_INVALID_ARG, "context %lld + %d passes max_context %d", (long long)lh.length, n_new,
                    c->cfg.max_context);
    cudaError_t e = launch_append(lh.dev, c->cdev, layer, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, n_new,
                                  (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "append kernel");
    lh.length += n_new;
    note_op(c, layer, stream);
    return QEVICT_OK;
}

static qevict_status decode_common(qevict_cache *c, int32_t layer, const void *q, const void *k_new, const void *v_new,
                                   float *out, float *mass, int32_t accumulate, void *stream) {
    qevict_status st = check_layer(c, layer);
    if (st) return st;
    LayerHost &lh = c->layers[layer];
    if (!q || !out) return fail(QEVICT_ERR_INVALID_ARG, "q and out must not be NULL");
    if (k_new) {
        if (lh.length + 1 > c->cfg.max_context)
            return fail(QEVICT_ERR_INVALID_ARG, "context %lld + 1 passes max_context %d", (long long)lh.length,
                        c->cfg.max_context);
    } else if (lh.length < 1) {
        return fail(QEVICT_ERR_INVALID_ARG, "layer %d is empty", layer);
    }
    const int splits = decode_splits(c->cfg.batch * c->cfg.num_kv_heads, c->num_sms, c->G);
    const bool pdl = c->allow_pdl && c->prev_layer >= 0 && c->prev_layer != layer && c->prev_stream == stream;
    cudaError_t e = launch_decode(lh.dev, c->cdev, c->scratch, lh.tmap, layer, (const __nv_bfloat16 *)q,
                                  (const __nv_bfloat16 *)k_new, (const __nv_bfloat16 *)v_new, out, mass,
                                  accumulate, splits, pdl, c->coop, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel");
    if (k_new) lh.length += 1;
    return QEVICT_OK;
}

qevict_status qevict_decode_attention(qevict_cache *c, int32_t layer, const void *q, float *out, float *mass,
                                      int32_t accumulate_scores, void *stream) {
    qevict_status st = decode_common(c, layer, q, nullptr, nullptr, out, mass, accumulate_scores, stream);
    if (!st) note_op(c, layer, stream);
    return st;
}

qevict_status qevict_decode_step(qevict_cache *c, int32_t layer, const void *q, const void *k_new, const void *v_new,
                                 float *out, float *mass, int32_t accumulate_scores, void *stream) {
    if (!k_new || !v_new) return fail(QEVICT_ERR_INVALID_ARG, "k_new and v_new must not be NULL");
    qevict_status st = decode_common(c, layer, q, k_new, v_new, out, mass, accumulate_scores, stream);
    if (!st) note_op(c, layer, stream);
    return st;
}

qevict_status qevict_route_rd(qevict_cache *c, int32_t layer, const float *scores_override, const float *score_mult,
                              void *stream) {
    qevict_status st = check_layer(c, layer);
    if (st) return st;
    st = check_int2_only(c, "the rate-distortion route");
    if (st) return st;
    LayerHost &lh = c->layers[layer];
    if (lh.length == 0) return QEVICT_OK;
    const int64_t Bt = budget_bytes(c->cfg, lh.length);
    if (Bt < c->c_fp)
        return fail(QEVICT_ERR_BUDGET, "budget %lld B cannot hold the open window (%lld B)", (long long)Bt,
                    (long long)c->c_fp);
    PlanArgs a{};
    a.mode = PLAN_RD;
    a.layer = layer;
    a.scores = scores_override;
    a.mult = score_mult;
    return run_plan(c, lh, a, nullptr, nullptr, (cudaStream_t)stream);
}

qevict_status qevict_k_channel_weights(qevict_cache *c, int32_t layer, const void *q_obs, int64_t n_q,
                                      const void *k_full, int64_t n_tokens, float *weights, void *stream) {
    qevict_status st = check_layer(c, layer);
    if (st) return st;
    if (!q_obs || !k_full || !weights) return fail(QEVICT_ERR_INVALID_ARG, "q_obs, k_full and weights must be set");
    if (n_q < 1 || n_tokens < 1 || n_q > INT32_MAX)
        return fail(QEVICT_ERR_INVALID_ARG, "n_q (%lld) and n_tokens (%lld) must be positive", (long long)n_q,
                    (long long)n_tokens);
    if (c->hs != 1) return fail(QEVICT_ERR_INVALID_ARG, "K-channel weights need shared tiers (not per KV head)");
    if (((uintptr_t)q_obs | (uintptr_t)k_full) & 15)
        return fail(QEVICT_ERR_INVALID_ARG, "q_obs and k_full must be 16-byte aligned");
    cudaError_t e = launch_k_channel_weights(c->layers[layer].dev, (const __nv_bfloat16 *)q_obs, (int)n_q,
                                             (const __nv_bfloat16 *)k_full, n_tokens, weights, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "K channel weights kernel");
    note_op(c, -1, stream);
    return QEVICT_OK;
}

qevict_status qevict_route_rd_kv(qevict_cache *c, int32_t layer, const float *weights, const float *scores_override,
                                 void *stream) {
    qevict_status st = check_layer(c, layer);
    if (st) return st;
    if (!weights) return fail(QEVICT_ERR_INVALID_ARG, "weights must be set");
    if (c->cfg.max_ledger_bits != 8)
        return fail(QEVICT_ERR_INVALID_ARG, "K-channel routing needs max_ledger_bits 8 (this cache: %d)",
                    c->cfg.max_ledger_bits);
    if (c->hs != 1) return fail(QEVICT_ERR_INVALID_ARG, "K-channel routing needs shared tiers (not per KV head)");
    if (c->cfg.num_kv_heads > 16) return fail(QEVICT_ERR_INVALID_ARG, "K-channel routing takes at most 16 KV heads");
    LayerHost &lh = c->layers[layer];
    if (lh.kch) return fail(QEVICT_ERR_STATE, "layer %d already has its K-channel widths", layer);
    if (lh.length == 0) return QEVICT_OK;
    const int64_t Bt = budget_bytes(c->cfg, lh.length);
    if (Bt < c->c_fp)
        return fail(QEVICT_ERR_BUDGET, "budget %lld B cannot hold the open window (%lld B)", (long long)Bt,
                    (long long)c->c_fp);
    PlanArgs a{};
    a.mode = PLAN_RD_KV;
    a.layer = layer;
    a.scores = scores_override;
    a.kweights = weights;
    lh.kch = true;
    return run_plan(c, lh, a, nullptr, nullptr, (cudaStream_t)stream);
}

qevict_status qevict_route_rd_mixed(qevict_cache *c, int32_t layer, const float *scores_override,
                                    const float *score_mult, void *stream) {
    qevict_status st = check_layer(c, layer);
    if (st) return st;
    LayerHost &lh = c->layers[layer];
    if (lh.length == 0) return QEVICT_OK;
    const int64_t Bt = budget_bytes(c->cfg, lh.length);
    if (Bt < c->c_fp)
        return fail(QEVICT_ERR_BUDGET, "budget %lld B cannot hold the open window (%lld B)", (long long)Bt,
                    (long long)c->c_fp);
    PlanArgs a{};
    a.mode = PLAN_RD_MIXED;
    a.layer = layer;
    a.scores = scores_override;
    a.mult = score_mult;
    return run_plan(c, lh, a, nullptr, nullptr, (cudaStream_t)stream);
}

qevict_status qevict_route_logsparse(qevict_cache *c, int32_t layer, int32_t recent_windows, void *stream) {
    qevict_status st = check_layer(c, layer);
    if (st) return st;
    st = check_int2_only(c, "the log-sparse route");
    if (st) return st;
    if (recent_windows < 1) return fail(QEVICT_ERR_INVALID_ARG, "recent_windows must be >= 1");
    LayerHost &lh = c->layers[layer];
    if (lh.length == 0) return QEVICT_OK;
    const int64_t Bt = budget_bytes(c->cfg, lh.length);
    if (Bt < c->c_fp)
        return fail(QEVICT_ERR_BUDGET, "budget %lld B cannot hold the open window (%lld B)", (long long)Bt,
                    (long long)c->c_fp);
    PlanArgs a{};
    a.mode = PLAN_LOGSPARSE;
    a.layer = layer;
    a.recent = recent_windows;
    return run_plan(c, lh, a, nullptr, nullptr, (cudaStream_t)stream);
}

qevict_status qevict_route_global(qevict_cache *c, const float *const *scores_override, void *stream) {
    if (!c) return fail(QEVICT_ERR_INVALID_ARG, "cache is NULL");
    {
        const qevict_status st = check_int2_only(c, "the global route");
        if (st) return st;
    }
    const qevict_config &cfg = c->cfg;
    cudaStream_t s = (cudaStream_t)stream;
    // host check of the one budget against the forced windows (host lengths)
    int64_t F = 0;
    int forced = 0;
    for (int l = 0; l < cfg.num_layers; ++l) {
        F += (int64_t)c->hs * c->layers[l].length * cfg.num_kv_heads * kHeadDim * 4;
        forced += c->layers[l].length > 0 ? c->hs : 0;
    }
    if (forced == 0) return QEVICT_OK;
    if (cfg.batch / c->hs > 65535) return fail(QEVICT_ERR_INVALID_ARG, "a global event takes at most 65535 sequences");
    const int64_t Bg = (int64_t)floor(cfg.budget_frac * (double)F);
    if ((int64_t)forced * c->c_fp > Bg)
        return fail(QEVICT_ERR_BUDGET, "budget %lld B cannot hold the %d open windows (%lld B each)", (long long)Bg,
                    forced, (long long)c->c_fp);
    cudaError_t e = cudaSuccess;
    if (scores_override)
        for (int l = 0; l < cfg.num_layers && e == cudaSuccess; ++l)
            if (scores_override[l] && c->layers[l].length > 0)
                e = launch_set_scores(c->layers[l].dev, scores_override[l], n_windows(c, c->layers[l].length), s);
    if (e != cudaSuccess) return cuda_fail(e, "score override kernel");
    GlobalArgs g{};
    g.layers = c->ldev;
    g.num_layers = cfg.num_layers;
    g.hs = c->hs;
    g.Wmax = c->Wmax;
    g.w = cfg.window;
    g.beta = cfg.budget_frac;
    g.rho = cfg.fp_share;
    g.c_fp = c->c_fp;
    g.c_q = c->c_q;
    g.keys = c->gkeys;
    g.thr = c->gthr;
    g.flag = c->gflag;
    g.cnt = c->gcnt;
    e = launch_global_select(g, c->cdev, cfg.batch / c->hs, s);
    if (e != cudaSuccess) return cuda_fail(e, "global select kernel");
    for (int l = 0; l < cfg.num_layers; ++l) {
        LayerHost &lh = c->layers[l];
        if (lh.length == 0) continue;
        PlanArgs a{};
        a.mode = PLAN_GLOBAL;
        a.layer = l;
        a.gkeys = c->gkeys;
        a.gthr = c->gthr;
        a.gflag = c->gflag;
        a.glayers = cfg.num_layers;
        const qevict_status st = run_plan(c, lh, a, nullptr, nullptr, s);
        if (st) return st;
    }
    return QEVICT_OK;
}

qevict_status qevict_route(qevict_cache *c, int32_t layer, const float *scores_override, const float *score_mult,
                           void *stream) {
    qevict_status st = check_layer(c, layer);
    if (st) return st;
    st = check_int2_only(c, "the score route");
    if (st) return st;
    LayerHost &lh = c->layers[layer];
    if (lh.length == 0) return QEVICT_OK;
    PlanArgs a{};
    a.mode = PLAN_ROUTE;
    a.layer = layer;
    a.scores = scores_override;
    a.mult = score_mult;
    const int64_t Bt = budget_bytes(c->cfg, lh.length);
    if (Bt < c->c_fp)
        return fail(QEVICT_ERR_BUDGET, "budget %lld B cannot hold the open window (%lld B)", (long long)Bt,
                    (long long)c->c_fp);
    return run_plan(c, lh, a, nullptr, nullptr, (cudaStream_t)stream);
}

static qevict_status listed(qevict_cache *c, int32_t layer, const int32_t *bw, int32_t n, int mode, void *stream) {
    qevict_status st = check_layer(c, layer);
    if (st) return st;
    LayerHost &lh = c->layers[layer];
    if (n < 0) return fail(QEVICT_ERR_INVALID_ARG, "n must be >= 0");
    if (n == 0 || lh.length == 0) return QEVICT_OK;
    if (!bw) return fail(QEVICT_ERR_INVALID_ARG, "bw_ids must not be NULL");
    PlanArgs a{};
    a.mode = mode;
    a.layer = layer;
    a.pairs = bw;
    a.n_pairs = n;
    return run_plan(c, lh, a, nullptr, nullptr, (cudaStream_t)stream);
}

qevict_status qevict_demote_quantize(qevict_cache *c, int32_t layer, const int32_t *bw_ids, int32_t n, void *stream) {
    return listed(c, layer, bw_ids, n, PLAN_DEMOTE, stream);
}

qevict_status qevict_promote_dequantize(qevict_cache *c, int32_t layer, const int32_t *bw_ids, int32_t n,
                                        void *stream) {
    return listed(c, layer, bw_ids, n, PLAN_PROMOTE, stream);
}

qevict_status qevict_set_tiers(qevict_cache *c, int32_t layer, const uint8_t *tiers, void *stream) {
    qevict_status st = check_layer(c, layer);
    if (st) return st;
    LayerHost &lh = c->layers[layer];
    if (!tiers) return fail(QEVICT_ERR_INVALID_ARG, "tiers must not be NULL");
    if (lh.length == 0) return QEVICT_OK;
    PlanArgs a{};
    a.mode = PLAN_TIERS;
    a.layer = layer;
    a.tiers = tiers;
    return run_plan(c, lh, a, nullptr, nullptr, (cudaStream_t)stream);
}

qevict_status qevict_get_scores(qevict_cache *c, int32_t layer, float *scores, void *stream) {
    qevict_status st = check_layer(c, layer);
    if (st) return st;
    if (!scores) return fail(QEVICT_ERR_INVALID_ARG, "scores must not be NULL");
    LayerHost &lh = c->layers[layer];
    const int nw = n_windows(c, lh.length);
    if (nw == 0) return QEVICT_OK;
    cudaError_t e = launch_scores(lh.dev, nw, scores, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "scores kernel");
    note_op(c, layer, stream);
    return QEVICT_OK;
}

qevict_status qevict_get_view(const qevict_cache *c, int32_t layer, qevict_view *v) {
    qevict_status st = check_layer(c, layer);
    if (st) return st;
    if (!v) return fail(QEVICT_ERR_INVALID_ARG, "view must not be NULL");
    const LayerHost &lh = c->layers[layer];
    const LayerDev &D = lh.dev;
    v->batch = D.B;
    v->num_q_heads = D.Hq;
    v->num_kv_heads = D.Hkv;
    v->head_dim = kHeadDim;
    v->window = D.w;
    v->max_windows = D.Wmax;
    v->num_windows = n_windows(c, lh.length);
    v->fp_capacity = D.CF;
    v->ledger_capacity = D.CQ;
    v->length = lh.length;
    v->fp_slot_bytes = D.fp_slot_bytes;
    v->ledger_slot_bytes = D.lg_slot_bytes;
    v->tier = D.tier;
    v->fp_slot = D.fp_slot;
    v->ledger_slot = D.lg_slot;
    v->ledger_writes = D.lwrites;
    v->fp_pool = D.fp_pool;
    v->ledger_pool = D.lg_pool;
    v->ledger_bits = D.lbits;
    v->max_ledger_bits = 2 * D.maxP;
    v->k_group_bits = lh.kch ? D.kgw : nullptr;
    return QEVICT_OK;
}

qevict_status qevict_get_status(qevict_cache *c, void *stream) {
    if (!c) return fail(QEVICT_ERR_INVALID_ARG, "cache is NULL");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronise");
    int32_t s[4];
    e = cudaMemcpy(s, c->cdev.status, sizeof s, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "status copy");
    if (s[0] != 0) {
        g_last_error = "device status " + std::to_string(s[0]) + " at layer " + std::to_string(s[1]) +
                       " (sequence " + std::to_string(s[2]) + ", item " + std::to_string(s[3]) + ")";
    }
    return (qevict_status)s[0];
}

qevict_status qevict_clear_status(qevict_cache *c, void *stream) {
    if (!c) return fail(QEVICT_ERR_INVALID_ARG, "cache is NULL");
    cudaError_t e = cudaMemsetAsync(c->cdev.status, 0, 16, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "status reset");
    // A decode that gave up waiting may leave tagged split records and counters
    // behind that a later launch would take for its own: start them afresh.
    uint8_t *sb = reinterpret_cast<uint8_t *>(c->scratch_base);
    if (sb) {
        const size_t n0 = (size_t)(reinterpret_cast<uint8_t *>(c->scratch.rec) - sb);
        const size_t o1 = (size_t)(reinterpret_cast<uint8_t *>(c->scratch.bar) - sb);
        e = cudaMemsetAsync(sb, 0, n0, (cudaStream_t)stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(sb + o1, 0, c->scratch_bytes - o1, (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "decode scratch reset");
    }
    note_op(c, -1, stream);
    return QEVICT_OK;
}

qevict_status qevict_set_cooperative_launch(qevict_cache *c, int32_t enable) {
    if (!c) return fail(QEVICT_ERR_INVALID_ARG, "cache is NULL");
    c->coop = enable != 0;
    return QEVICT_OK;
}

qevict_status qevict_set_wait_limit(qevict_cache *c, int64_t cycles) {
    if (!c) return fail(QEVICT_ERR_INVALID_ARG, "cache is NULL");
    c->cdev.wait_cycles = cycles > 0 ? (long long)cycles : kDefaultWaitCycles;
    return QEVICT_OK;
}

qevict_status qevict_get_stats(qevict_cache *c, qevict_stats *out, void *stream) {
    if (!c || !out) return fail(QEVICT_ERR_INVALID_ARG, "cache and stats must not be NULL");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronise");
    unsigned long long s[ST_N];
    e = cudaMemcpy(s, c->cdev.stats, sizeof s, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "stats copy");
    out->demotions = s[ST_DEMOTE];
    out->promotions = s[ST_PROMOTE];
    out->evictions = s[ST_EVICT];
    out->ledger_writes = s[ST_LWRITE];
    out->ledger_reuses = s[ST_LREUSE];
    out->device_bytes = c->total_bytes;
    return QEVICT_OK;
}

qevict_status qevict_get_tier_move_counts(qevict_cache *c, int32_t layer, int32_t *counts, void *stream) {
    qevict_status st = check_layer(c, layer);
    if (st) return st;
    if (!counts) return fail(QEVICT_ERR_INVALID_ARG, "counts must not be NULL");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e == cudaSuccess)
        e = cudaMemcpy(counts, c->layers[layer].dev.diag, (size_t)c->cfg.batch * 8 * sizeof(int32_t),
                       cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "tier move counts copy");
    return QEVICT_OK;
}

qevict_status qevict_future_missed_mass(qevict_cache *c, int32_t layer, const void *q, const void *k_full,
                                        int64_t n_tokens, float *fmm, void *stream) {
    qevict_status st = check_layer(c, layer);
    if (st) return st;
    if (!q || !k_full || !fmm) return fail(QEVICT_ERR_INVALID_ARG, "q, k_full and fmm must not be NULL");
    if (((uintptr_t)q | (uintptr_t)k_full) & 15) return fail(QEVICT_ERR_INVALID_ARG, "q and k_full must be 16-byte aligned");
    LayerHost &lh = c->layers[layer];
    if (lh.length < 1) return fail(QEVICT_ERR_INVALID_ARG, "layer %d is empty", layer);
    if (n_tokens != lh.length)
        return fail(QEVICT_ERR_INVALID_ARG, "n_tokens %lld differs from the layer's length %lld", (long long)n_tokens,
                    (long long)lh.length);
    if ((int64_t)c->cfg.batch * n_tokens > INT32_MAX)
        return fail(QEVICT_ERR_INVALID_ARG, "batch x n_tokens passes 2^31 - 1");
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return fail(QEVICT_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    // k_full as [sequences * n_tokens][model KV heads][128]: boxes of 64 channels x 1 KV head x 16 tokens
    CUtensorMap kmap{};
    const int hs = lh.dev.hs;
    const cuuint64_t heads = (cuuint64_t)c->cfg.num_kv_heads * hs;
    const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, heads, (cuuint64_t)(c->cfg.batch / hs) * (cuuint64_t)n_tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, heads * kHeadDim * 2};
    const cuuint32_t box[3] = {64, 1, 16};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(k_full), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return fail(QEVICT_ERR_INVALID_ARG, "k_full cannot be described as a tensor map");
    cudaError_t e = launch_future_missed_mass(lh.dev, c->cdev, c->scratch, layer, kmap, (const __nv_bfloat16 *)q,
                                              (int)n_tokens, fmm, c->num_sms, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "future missed mass kernels");
    note_op(c, layer, stream);
    return QEVICT_OK;
}

qevict_status qevict_set_launch_overlap(qevict_cache *c, int32_t enable) {
    if (!c) return fail(QEVICT_ERR_INVALID_ARG, "cache is NULL");
    c->allow_pdl = enable != 0;
    return QEVICT_OK;
}

qevict_status qevict_refresh_lengths(qevict_cache *c, void *stream) {
    if (!c) return fail(QEVICT_ERR_INVALID_ARG, "cache is NULL");
    cudaStream_t s = (cudaStream_t)stream;
    int32_t *dbuf = reinterpret_cast<int32_t *>((uint8_t *)c->cbase + 128);
    for (int l = 0; l < c->cfg.num_layers; ++l) {
        cudaError_t e = launch_read_lengths(c->layers[l].dev, dbuf, s);
        int32_t len = 0;
        if (e == cudaSuccess) e = cudaMemcpyAsync(&len, dbuf, sizeof len, cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e, "length refresh");
        c->layers[l].length = len;
    }
    return QEVICT_OK;
}

int64_t qevict_length(const qevict_cache *c, int32_t layer) {
    if (!c || layer < 0 || layer >= c->cfg.num_layers) return -1;
    return c->layers[layer].length;
}

}  // extern "C"

// ---- decode with library-owned static scratch ------------------------------
// The decode needs per-call scratch (split partials, records, chunk records
// and the split arrival counters). qevict_decode_attention_static_scratch takes it from the
// fixed device array below instead of the cache's own block, so the call
// allocates nothing. Its address is looked up once per device, with that
// device current, and then passed to the kernel as a plain pointer.

namespace {

constexpr size_t kStaticScratchBytes = QEVICT_STATIC_SCRATCH_BYTES;
constexpr int kStaticMaxDevices = 64;

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void *g_static_ptr[kStaticMaxDevices];

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// Scratch layout of one call: split arrival counters and record generations,
// the tagged split records and partials, then the chunk records. The offsets
// depend on the cache's shape, so one cache's counters could lie on another's
// records: every call clears everything before the chunk records on its
// stream first (a memset, which allocates nothing). After the clear the
// record generation is 0, so the launch's tag is 1 and no word left by an
// earlier call carries it. The chunk records are written before they are read.
struct StaticLayout {
    size_t o_bar, o_stat, o_part, o_rec, total;
    int rec_stride;
};

StaticLayout static_layout(const qevict_cache *c, int splits) {
    const size_t B = (size_t)c->cfg.batch, Hkv = (size_t)c->cfg.num_kv_heads;
    const int maxP = c->cfg.max_ledger_bits > 2 ? c->cfg.max_ledger_bits / 2 : 1;
    StaticLayout s{};
    s.rec_stride = decode_records(c->CF, c->CQ, c->cfg.window, maxP);
    s.o_bar = 0;
    s.o_stat = s.o_bar + round256(B * Hkv * 8);
    s.o_part = s.o_stat + round256(B * Hkv * (size_t)kMaxSplits * kMaxG * 16);
    s.o_rec = s.o_part + round256(B * Hkv * (size_t)splits * c->G * kHeadDim * 8);
    s.total = s.o_rec + round256(B * Hkv * (size_t)s.rec_stride * c->G * 8);
    return s;
}

// First use on a device: look up the array's address (and clear the array once).
qevict_status static_scratch_setup(int dev, void **out) {
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "static scratch address lookup");
        e = cudaMemset(p, 0, kStaticScratchBytes);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "static scratch clear");
        g_static_ptr[dev] = p;
    }
    *out = g_static_ptr[dev];
    return QEVICT_OK;
}

}  // namespace

extern "C" {

qevict_status qevict_decode_attention_static_scratch(qevict_cache *c, int32_t layer, const void *q, float *out,
                                                     float *mass, int32_t accumulate_scores, void *stream) {
    qevict_status st = check_layer(c, layer);
    if (st) return st;
    LayerHost &lh = c->layers[layer];
    if (!q || !out) return fail(QEVICT_ERR_INVALID_ARG, "q and out must not be NULL");
    if (lh.length < 1) return fail(QEVICT_ERR_INVALID_ARG, "layer %d is empty", layer);
    const int splits = decode_splits(c->cfg.batch * c->cfg.num_kv_heads, c->num_sms, c->G);
    const StaticLayout ly = static_layout(c, splits);
    if (ly.total > kStaticScratchBytes)
        return fail(QEVICT_ERR_INVALID_ARG,
                    "this cache needs %zu B of decode scratch; the static scratch holds %zu B "
                    "(use qevict_decode_attention)",
                    ly.total, kStaticScratchBytes);
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != c->device)
        return fail(QEVICT_ERR_INVALID_ARG, "device %d is current but the cache lives on device %d", dev, c->device);
    if (dev < 0 || dev >= kStaticMaxDevices)
        return fail(QEVICT_ERR_INVALID_ARG, "device index %d passes the static scratch table (%d)", dev,
                    kStaticMaxDevices);
    void *base = nullptr;
    st = static_scratch_setup(dev, &base);
    if (st) return st;
    uint8_t *p = (uint8_t *)base;
    DecodeScratch S{};
    S.bar = (uint32_t *)(p + ly.o_bar);
    S.stat = (unsigned long long *)(p + ly.o_stat);
    S.part = (unsigned long long *)(p + ly.o_part);
    S.rec = (float2 *)(p + ly.o_rec);
    S.rec_stride = ly.rec_stride;
    e = cudaMemsetAsync(p, 0, ly.o_rec, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "static scratch clear");
    e = launch_decode(lh.dev, c->cdev, S, lh.tmap, layer, (const __nv_bfloat16 *)q, nullptr, nullptr, out, mass,
                      accumulate_scores, splits, false, c->coop, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel");
    note_op(c, layer, stream);
    return QEVICT_OK;
}

}  // extern "C"
