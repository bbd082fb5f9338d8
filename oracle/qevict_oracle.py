"""Plain CPU oracle of QEvict's recoverable three-tier KV cache on the decode path.

TEST INFRASTRUCTURE. Only the test-suite, the smoke check and the benchmark's
CPU-baseline leg import this module. The library (C-ABI + CUDA kernels) never
calls it, and this module imports nothing from the library.

What it follows, cited by page title and section:

* "Technische Samenvatting: QEvict" (gist.science/nl/paper/2608.05326) and its
  Chinese twin (gist.science/zh/paper/2608.05326), sections "Methodologie:
  QEvict" (three tiers: full precision, recoverable INT2, evicted; a fixed
  byte budget) and "Kernmechanismen" (window-level routing, cumulative
  scoring, demotion, promotion, the write-once quantisation ledger, GQA).
* "Technische Samenvatting: LogQuant" (gist.science/nl/paper/2503.19950),
  Methodologie 3 (evicting a token removes it from the softmax normalisation)
  and 4 (the order of cache entries does not change A.V).
* "Technische Samenvatting: RDKV" (gist.science/nl/paper/2605.08317), 2.1
  (the importance of a token is the attention mass it receives, summed over
  queries).

The pages give no formulas for QEvict's quantiser or router. Where they are
silent this module takes the plainest reading (one tier per window shared by
all KV heads, asymmetric min/max INT2 over groups of 32 channels with fp16
scale and minimum, window score = mean over query heads of the window's
softmax mass, budget counts only attention-visible bytes, the last window is
always full precision, FP share of the budget rho). Each reading is named
where it is used.

Floating point: attention, masses and scores in float64. The quantiser and the
promotion dequantiser are integer-producing / rounding steps whose results must
match bit for bit, so they are written in the exact float32 / float16
operations they are defined by (numpy float32 arithmetic and float32 ->
float16 casts are IEEE round-to-nearest-even).

Parity status: attention/masses/scores pinned by the dense-softmax special
case, mass sums, closed forms and brute force; quantiser pinned by exact-grid
groups, nearest-level optimality and the error bound; router pinned by brute
force over all tier assignments on small inputs. Nothing here is "parity
unpinned".
"""
from __future__ import annotations

import math

import numpy as np

TIER_FP, TIER_Q, TIER_E = 0, 1, 2
TIER_Q4, TIER_Q8 = 3, 4   # the 4- and 8-bit widths of the rate-distortion option (RDKV 2.2)
GROUP = 32          # channels per INT2 quantisation group
LEVELS = 3          # 2-bit codes 0..3 -> (max - min) / 3 per step
BITS_OF_TIER = {TIER_Q: 2, TIER_Q4: 4, TIER_Q8: 8}
TIER_OF_BITS = {0: TIER_E, 2: TIER_Q, 4: TIER_Q4, 8: TIER_Q8, 16: TIER_FP}


class OracleError(Exception):
    """Base of the oracle's error conditions (mirrors the library's status codes)."""


class BudgetError(OracleError):
    pass


class StateError(OracleError):
    pass


class QuantError(OracleError):
    pass


# --------------------------------------------------------------------------
# Exact rounding helpers
# --------------------------------------------------------------------------

def bf16_round(x) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32.

    bfloat16 keeps the top 16 bits of a float32. Adding 0x7FFF plus the lowest
    kept bit to the 32-bit pattern and truncating rounds the dropped 16 bits to
    nearest, ties to the even kept value; an overflow out of the largest finite
    value carries into the exponent and yields infinity, as IEEE rounding does.
    NaN stays NaN.
    """
    x = np.asarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    out = r.astype(np.uint32).view(np.float32)
    return np.where(np.isnan(x), x, out).astype(np.float32)


def half_round(x) -> np.ndarray:
    """Round float32 values to float16 (IEEE round-to-nearest-even, with subnormals)."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float32).astype(np.float16)


# --------------------------------------------------------------------------
# INT2 quantiser (demotion) and dequantisers
# --------------------------------------------------------------------------

def quantize_groups(x, bits: int = 2):
    """Asymmetric 2-bit (or, for the mixed-width option, 4- or 8-bit)
    quantisation of groups of 32 bf16 values.

    Reading of QEvict "Recoverable Quantized Tier" (INT2): per token, per KV
    head, per group of 32 consecutive channels of head_dim, for K and V alike:

      mn = min x, mx = max x                               (exact)
      min16   = fp16_rne(mn)
      scale16 = fp16_rne(fl32(fl32(mx - mn) / 3))
      code_j  = clamp(rint_even(fl32(fl32(x_j - min16) / scale16)), 0, 3)
                (all codes 0 when scale16 == 0)

    With ``bits`` b the 3 above is 2^b - 1 (RDKV 2.2: widths 2, 4, 8 of one
    scheme; the pages give no other rule).

    x: float32 array [..., 32] holding bf16 values.
    Returns (codes uint8 [..., 32], scale float16 [...], minimum float16 [...],
    bad bool [...]) where ``bad`` flags a group with a non-finite input or a
    scale / minimum that overflows fp16 (the library reports these as a status
    error and leaves the group's codes at 0).
    """
    x = np.asarray(x, dtype=np.float32)
    assert x.shape[-1] == GROUP and bits in (2, 4, 8)
    levels = (1 << bits) - 1
    finite = np.isfinite(x).all(axis=-1)
    xs = np.where(np.isfinite(x), x, np.float32(0))
    mn = xs.min(axis=-1)
    mx = xs.max(axis=-1)
    mn16 = half_round(mn)
    with np.errstate(over="ignore", invalid="ignore"):
        rng = (mx - mn).astype(np.float32)
        s32 = (rng / np.float32(levels)).astype(np.float32)
    s16 = half_round(s32)
    bad = ~finite | ~np.isfinite(mn16) | ~np.isfinite(s16)
    s32q = s16.astype(np.float32)
    m32q = mn16.astype(np.float32)
    zero = (s32q == 0) | bad
    den = np.where(zero, np.float32(1), s32q)
    with np.errstate(over="ignore", invalid="ignore"):
        diff = (xs - m32q[..., None]).astype(np.float32)
        qt = (diff / den[..., None]).astype(np.float32)
    codes = np.clip(np.rint(qt), 0, levels)
    codes = np.where(zero[..., None], 0, codes).astype(np.uint8)
    s16 = np.where(bad, np.float16(0), s16)
    mn16 = np.where(bad, np.float16(0), mn16)
    return codes, s16.astype(np.float16), mn16.astype(np.float16), bad


def dequant_exact(codes, scale16, min16):
    """Real value min + code * scale of each code (float64, exact for fp16 meta).

    Used inside attention: the quantised tier is attended in place, without
    rounding the reconstruction.
    """
    c = np.asarray(codes, dtype=np.float64)
    s = np.asarray(scale16, dtype=np.float64)[..., None]
    m = np.asarray(min16, dtype=np.float64)[..., None]
    return m + c * s


def dequant_promote(codes, scale16, min16):
    """Promotion back to the full-precision tier: bf16_rne(fl32(code * scale + min)).

    code * scale + min is exact in float64 for fp16 scale / min and codes up to
    255 (an 8-bit code times an 11-bit significand, plus an fp16 value), so the
    float32 cast below is the single rounding of a fused multiply-add.
    """
    exact = dequant_exact(codes, scale16, min16)
    return bf16_round(exact.astype(np.float32))


# --------------------------------------------------------------------------
# Budget and routing
# --------------------------------------------------------------------------

def window_costs(w: int, Hkv: int, d: int):
    """Bytes one window occupies per sequence in each visible tier.

    full precision: K and V bf16, w * Hkv * d * 2 * 2;
    INT2: K and V codes (d / 4 bytes per token and head) plus one fp16 scale
    and one fp16 minimum per group of 32 channels.
    """
    c_fp = w * Hkv * d * 4
    c_q = w * Hkv * 2 * (d // 4 + 4 * (d // GROUP))
    return c_fp, c_q


def budget_bytes(L: int, Hkv: int, d: int, beta: float) -> int:
    """B_t = floor(beta * F_t), F_t = bytes of the full bf16 K/V cache at length L."""
    F = L * Hkv * d * 4
    return int(math.floor(beta * F))


def fp_budget_windows(Bt: int, c_fp: int, rho: float) -> int:
    """floor(rho * B_t / c_fp): full-precision windows the FP share of the budget buys."""
    return int(math.floor((rho * Bt) / c_fp))


def route_counts(n_cand: int, L: int, w: int, Hkv: int, d: int, beta: float, rho: float):
    """(n_fp, n_q) for one sequence at length L with n_cand non-evicted windows."""
    c_fp, c_q = window_costs(w, Hkv, d)
    Bt = budget_bytes(L, Hkv, d, beta)
    if Bt < c_fp:
        raise BudgetError(f"budget {Bt} B cannot hold the open window ({c_fp} B)")
    n_fp = min(n_cand, max(1, fp_budget_windows(Bt, c_fp, rho)))
    n_q = min(n_cand - n_fp, (Bt - n_fp * c_fp) // c_q)
    return n_fp, n_q


def route_tiers(S, tiers, L: int, w: int, Hkv: int, d: int, beta: float, rho: float):
    """Budgeted tier assignment for one sequence (QEvict "Kernmechanismen").

    Candidates are the windows that are not evicted (eviction is permanent).
    The last window (the one appends go into) is forced to full precision
    when it is a candidate. The rest are ranked by cumulative score, highest
    first, ties to the lower window index; the top n_fp (including the forced
    window) stay / become full precision, the next n_q INT2, the rest are
    evicted.
    Returns the new tier array (uint8).
    """
    W = -(-L // w)
    tiers = np.asarray(tiers, dtype=np.uint8)
    cand = [i for i in range(W) if tiers[i] != TIER_E]
    if not cand:
        return tiers.copy()
    vals = [float(S[i]) for i in cand]
    if not all(math.isfinite(v) for v in vals):
        raise OracleError("non-finite score among routing candidates")
    n_fp, n_q = route_counts(len(cand), L, w, Hkv, d, beta, rho)
    forced = W - 1
    order = sorted(cand, key=lambda i: (i != forced, -float(S[i]), i))
    new = tiers.copy()
    for r, i in enumerate(order):
        new[i] = TIER_FP if r < n_fp else (TIER_Q if r < n_fp + n_q else TIER_E)
    return new


# --------------------------------------------------------------------------
# Attention over the tiered cache
# --------------------------------------------------------------------------

def softmax_attention(q, keys, values):
    """o = softmax(q k^T / sqrt(d)) v for one head, in float64; also returns p."""
    q = np.asarray(q, dtype=np.float64)
    s = (np.asarray(keys, dtype=np.float64) @ q) / math.sqrt(q.shape[-1])
    s = s - s.max()
    e = np.exp(s)
    p = e / e.sum()
    return p @ np.asarray(values, dtype=np.float64), p


# --------------------------------------------------------------------------
# The cache as a state machine
# --------------------------------------------------------------------------

class Window:
    __slots__ = ("tier", "k", "v", "ledger", "ledger_bits", "ledger_writes", "ntok")

    def __init__(self, Hkv, w, d):
        self.tier = TIER_FP
        self.k = np.zeros((Hkv, w, d), np.float32)   # bf16 values
        self.v = np.zeros((Hkv, w, d), np.float32)
        self.ledger = None        # (codes_k, scale_k, min_k, codes_v, scale_v, min_v)
        self.ledger_bits = 0      # width of the ledger entry: 2, 4 or 8
        self.ledger_writes = 0
        self.ntok = 0


class OracleCache:
    """One layer of the tiered cache for a batch of B sequences of equal length."""

    def __init__(self, B, Hq, Hkv, d, w, beta=1.0, rho=0.5):
        assert Hq % Hkv == 0 and d % GROUP == 0
        self.B, self.Hq, self.Hkv, self.d, self.w = B, Hq, Hkv, d, w
        self.beta, self.rho = beta, rho
        self.L = 0
        self.win = [[] for _ in range(B)]
        self.S = [np.zeros(0, np.float64) for _ in range(B)]
        self.kch = None   # K-channel group widths [B][Hkv][4] once route_rd_kv has run
        self.kch_locked = False   # after it: no further tier moves (route_rd_kv)
        self.stats = dict(demotions=0, promotions=0, evictions=0, ledger_writes=0,
                          ledger_reuses=0)

    # ---- helpers --------------------------------------------------------
    @property
    def W(self):
        return -(-self.L // self.w)

    def tiers(self):
        return np.array([[win.tier for win in self.win[b]] for b in range(self.B)], np.uint8).reshape(self.B, self.W)

    def scores(self):
        return np.stack(self.S) if self.B else np.zeros((0, 0))

    # ---- appends (window partitioning) ------------------------------------
    def append(self, k, v):
        """Append n tokens' K, V ([B][n][Hkv][d], bf16 values) to every sequence.

        History is partitioned into consecutive windows of w tokens; a token at
        position p lands in window p // w, row p % w. A window opens in the
        full-precision tier when its first token arrives.
        """
        k = np.asarray(k, np.float32)
        v = np.asarray(v, np.float32)
        n = k.shape[1]
        for i in range(n):
            p = self.L + i
            wi, row = divmod(p, self.w)
            for b in range(self.B):
                if row == 0:
                    self.win[b].append(Window(self.Hkv, self.w, self.d))
                    self.S[b] = np.append(self.S[b], 0.0)
                win = self.win[b][wi]
                if win.tier != TIER_FP:
                    raise StateError("append into a window that is not full precision")
                win.k[:, row, :] = k[b, i]
                win.v[:, row, :] = v[b, i]
                win.ntok = row + 1
        self.L += n

    # ---- transitions (recoverable hierarchy + ledger) ----------------------
    def _evict(self, b, wi):
        win = self.win[b][wi]
        win.tier = TIER_E
        win.k = win.v = None
        win.ledger = None
        self.stats["evictions"] += 1

    def _demote(self, b, wi, tier=TIER_Q):
        """FP -> INT2 (or INT4 / INT8). Quantise only if the window has no
        ledger entry yet. The write-once ledger fixes a window's width at its
        first quantisation: a later demotion reuses the entry and must ask for
        the same width (re-quantising promoted values at another width would
        compound rounding, which the ledger exists to prevent)."""
        win = self.win[b][wi]
        if win.tier != TIER_FP or win.ntok != self.w:
            raise StateError("demotion needs a full full-precision window")
        bits = BITS_OF_TIER[tier]
        if win.ledger is None:
            if self.kch is None:
                ck, sk, mk, bk = quantize_groups(win.k.reshape(self.Hkv, self.w, -1, GROUP), bits)
            else:   # K groups at their channel widths (route_rd_kv)
                ck, sk, mk, bk = quantize_k_groups(win.k.reshape(self.Hkv, self.w, -1, GROUP), self.kch[b])
            cv, sv, mv, bv = quantize_groups(win.v.reshape(self.Hkv, self.w, -1, GROUP), bits)
            if bk.any() or bv.any():
                raise QuantError("non-finite value or fp16 overflow in a quantisation group")
            win.ledger = (ck.reshape(self.Hkv, self.w, self.d), sk, mk,
                          cv.reshape(self.Hkv, self.w, self.d), sv, mv)
            win.ledger_bits = bits
            win.ledger_writes += 1
            self.stats["ledger_writes"] += 1
        elif win.ledger_bits != bits:
            raise StateError("a window's quantised width is fixed by its first quantisation")
        else:
            self.stats["ledger_reuses"] += 1
        win.tier = tier
        win.k = win.v = None
        self.stats["demotions"] += 1

    def _promote(self, b, wi):
        """INT2 (INT4, INT8) -> FP: dequantise the ledger codes to bf16; the
        ledger is kept."""
        win = self.win[b][wi]
        if win.tier not in BITS_OF_TIER:
            raise StateError("promotion needs a quantised window")
        ck, sk, mk, cv, sv, mv = win.ledger
        g = lambda c: c.reshape(self.Hkv, self.w, -1, GROUP)
        win.k = dequant_promote(g(ck), sk, mk).reshape(self.Hkv, self.w, self.d)
        win.v = dequant_promote(g(cv), sv, mv).reshape(self.Hkv, self.w, self.d)
        win.tier = TIER_FP
        self.stats["promotions"] += 1

    def apply_tiers(self, b, new):
        """Move sequence b's windows to tiers ``new``: evict, then demote, then promote."""
        if self.kch_locked:
            raise StateError("a layer with K-channel widths takes no further tier moves")
        cur = [win.tier for win in self.win[b]]
        for wi, (c, t) in enumerate(zip(cur, new)):
            if c == TIER_E and t != TIER_E:
                raise StateError("an evicted window cannot come back")
            if c in BITS_OF_TIER and t in BITS_OF_TIER and c != t:
                raise StateError("a quantised window keeps its width")
            if c != t and wi == self.W - 1 and self.win[b][wi].ntok < self.w:
                raise StateError("the partially filled last window stays full precision")
        for wi, (c, t) in enumerate(zip(cur, new)):
            if c != TIER_E and t == TIER_E:
                self._evict(b, wi)
        for wi, (c, t) in enumerate(zip(cur, new)):
            if c == TIER_FP and t in BITS_OF_TIER:
                self._demote(b, wi, t)
        for wi, (c, t) in enumerate(zip(cur, new)):
            if c in BITS_OF_TIER and t == TIER_FP:
                self._promote(b, wi)

    def tiers_now(self, b):
        return [win.tier for win in self.win[b]]

    def set_tiers(self, tiers):
        tiers = np.asarray(tiers, np.uint8)
        counts = []
        for b in range(self.B):
            old = self.tiers_now(b)
            self.apply_tiers(b, tiers[b])
            counts.append(transition_counts(old, self.tiers_now(b)))
        self.last_counts = np.stack(counts)

    def route(self, scores_override=None, score_mult=None):
        """A routing event: optionally replace / scale the scores, rank, move tiers."""
        if scores_override is not None:
            ov = np.asarray(scores_override, np.float64)
            self.S = [ov[b, :self.W].copy() for b in range(self.B)]
        if score_mult is not None:
            mu = np.asarray(score_mult, np.float64)
            self.S = [self.S[b] * mu[b, :self.W] for b in range(self.B)]
        counts = []
        for b in range(self.B):
            old = self.tiers_now(b)
            new = route_tiers(self.S[b], old, self.L, self.w, self.Hkv, self.d, self.beta, self.rho)
            self.apply_tiers(b, new)
            counts.append(transition_counts(old, self.tiers_now(b)))
        self.last_counts = np.stack(counts)

    def prefill(self, k, v, scores=None, tiers=None):
        """Fill an empty cache with L tokens (all full precision), then route or set tiers."""
        assert self.L == 0
        self.append(k, v)
        if scores is not None:
            self.route(scores_override=scores)
        elif tiers is not None:
            self.set_tiers(tiers)

    def demote(self, pairs, tier=TIER_Q):
        if self.kch_locked:
            raise StateError("a layer with K-channel widths takes no further tier moves")
        old = [self.tiers_now(b) for b in range(self.B)]
        for b, wi in pairs:
            self._demote(b, wi, tier)
        self.last_counts = np.stack([transition_counts(old[b], self.tiers_now(b)) for b in range(self.B)])

    def promote(self, pairs):
        if self.kch_locked:
            raise StateError("a layer with K-channel widths takes no further tier moves")
        old = [self.tiers_now(b) for b in range(self.B)]
        for b, wi in pairs:
            self._promote(b, wi)
        self.last_counts = np.stack([transition_counts(old[b], self.tiers_now(b)) for b in range(self.B)])

    # ---- decode attention + cumulative scoring ----------------------------
    def window_kv(self, b, wi, kvh):
        """K, V rows (float64) a query attends to in window wi for KV head kvh, or None."""
        win = self.win[b][wi]
        if win.tier == TIER_E:
            return None
        n = win.ntok
        if win.tier == TIER_FP:
            return (win.k[kvh, :n].astype(np.float64), win.v[kvh, :n].astype(np.float64))
        ck, sk, mk, cv, sv, mv = win.ledger
        g = lambda c: c[kvh].reshape(self.w, -1, GROUP)
        kk = dequant_exact(g(ck), sk[kvh], mk[kvh]).reshape(self.w, self.d)
        vv = dequant_exact(g(cv), sv[kvh], mv[kvh]).reshape(self.w, self.d)
        return kk[:n], vv[:n]

    def decode(self, q, accumulate=True):
        """One decode step of single-token GQA attention over the tiered cache.

        q: [B][Hq][d] (bf16 values). Query head h reads KV head h // (Hq / Hkv).
        Full-precision windows are read as stored, INT2 windows as their exact
        reconstruction min + code * scale, evicted windows not at all (they
        leave the softmax denominator). Returns (out [B][Hq][d], mass
        [B][Hq][W]) in float64; mass[b, h, w] is the softmax probability the
        head puts on window w. With ``accumulate`` the window score grows by
        the mean of the masses over the Hq query heads.
        """
        q = np.asarray(q, np.float64)
        G = self.Hq // self.Hkv
        W = self.W
        out = np.zeros((self.B, self.Hq, self.d))
        mass = np.zeros((self.B, self.Hq, W))
        for b in range(self.B):
            for kvh in range(self.Hkv):
                ks, vs, owner = [], [], []
                for wi in range(W):
                    kv = self.window_kv(b, wi, kvh)
                    if kv is None:
                        continue
                    ks.append(kv[0])
                    vs.append(kv[1])
                    owner.append(np.full(kv[0].shape[0], wi))
                if not ks:
                    continue
                K = np.concatenate(ks)
                V = np.concatenate(vs)
                own = np.concatenate(owner)
                for h in range(kvh * G, (kvh + 1) * G):
                    o, p = softmax_attention(q[b, h], K, V)
                    out[b, h] = o
                    mass[b, h] = np.bincount(own, weights=p, minlength=W)
            if accumulate:
                self.S[b] = self.S[b] + mass[b].mean(axis=0)
        return out, mass


def transition_counts(old, new):
    """Diagnostics of one move of a sequence's tiers (QEvict, Kernbijdragen:
    selection churn and latent importance reactivation), with the full
    precision tier read as the active set:
    [fp_before, q_before, fp_after, q_after, kept, promoted, demoted, evicted],
    where kept counts windows full precision before and after, promoted INT2 ->
    full precision, demoted full precision -> INT2, evicted visible -> evicted.
    Selection churn = 1 - kept / fp_after; reactivation rate = promoted /
    q_before."""
    old = np.asarray(old)
    new = np.asarray(new)
    quant = lambda t: np.isin(t, list(BITS_OF_TIER))   # the recoverable tier, at any width
    return np.array([
        int((old == TIER_FP).sum()), int(quant(old).sum()),
        int((new == TIER_FP).sum()), int(quant(new).sum()),
        int(((old == TIER_FP) & (new == TIER_FP)).sum()),
        int((quant(old) & (new == TIER_FP)).sum()),
        int(((old == TIER_FP) & quant(new)).sum()),
        int(((old != TIER_E) & (new == TIER_E)).sum()),
    ], dtype=np.int64)


def future_missed_mass(cache, q, k_full):
    """Future missed mass (QEvict, Kernbijdragen): the share of a query's
    attention over the full, never-evicted cache that falls on windows the
    cache has evicted. q [B][Hq][d], k_full [B][L][Hkv][d] (the keys of all L
    tokens as stored before any tier move); returns [B][Hq] in float64."""
    q = np.asarray(q, np.float64)
    k_full = np.asarray(k_full, np.float64)
    B, L, Hkv, d = k_full.shape
    G = cache.Hq // Hkv
    out = np.zeros((B, cache.Hq))
    for b in range(B):
        tier_of_tok = np.array([cache.win[b][t // cache.w].tier for t in range(L)])
        for h in range(cache.Hq):
            s = k_full[b, :, h // G, :] @ q[b, h] / np.sqrt(d)
            p = np.exp(s - s.max())
            p /= p.sum()
            out[b, h] = p[tier_of_tok == TIER_E].sum()
    return out


# ---- per-KV-head tiers (an option) -------------------------------------------
#
# The default reading shares one tier per window between the KV heads. As an
# option each KV head keeps a cache of its own size ("Technische Samenvatting:
# DBTrimKV", Implementatie: head-specific cache sizes). Every (sequence, KV
# head) pair is then a unit routed on its own: its own windows and tiers, its
# own cumulative score (the mean mass of the G query heads that read it), and
# its own budget floor(beta * L * d * 4), the pair's share of the sequence's
# bytes. A query head attends only to its own KV head, so a unit is exactly a
# one-KV-head cache with G query heads, and that is how it is built here.

def per_head_cache(B, Hq, Hkv, d, w, beta=1.0, rho=0.5):
    """The per-head form of a cache of B sequences: B * Hkv units, unit
    u = b * Hkv + kvh, each with 1 KV head and Hq / Hkv query heads."""
    assert Hq % Hkv == 0
    return OracleCache(B * Hkv, Hq // Hkv, 1, d, w, beta, rho)


def to_units(x):
    """Token rows [B][n][Hkv][d] as unit rows [B * Hkv][n][1][d]."""
    x = np.asarray(x)
    B, n, H, d = x.shape
    return x.transpose(0, 2, 1, 3).reshape(B * H, n, 1, d)


def queries_to_units(q, Hkv):
    """Queries [B][Hq][d] as [B * Hkv][Hq / Hkv][d] (query head h reads KV head h // G)."""
    q = np.asarray(q)
    B, Hq, d = q.shape
    return q.reshape(B * Hkv, Hq // Hkv, d)


# ---- rate-distortion routing (an option) ------------------------------------
#
# "Technische Samenvatting: RDKV", 2.1-2.2: minimise sum_u w_u sigma_u 2^(-b_u)
# over bit widths b_u under a byte budget, solved by Lagrangian relaxation
# (reverse water-filling) over discrete widths. Here the units are windows,
# the widths the ones the tiers have (0 evicted, 2 INT2, 16 bf16), the weight
# w_u is the window's cumulative attention score (RDKV's weight of a V token
# is the attention it receives summed over queries) and sigma_u = 1. Each
# window has two upgrades: E -> INT2 removes 3/4 w_u of distortion for c_q
# bytes, INT2 -> FP removes (1/4 - 2^-16) w_u for c_fp - c_q bytes. The open
# window is full precision first; the other upgrades are taken in order of
# distortion removed per byte, highest first (E -> INT2 before INT2 -> FP on a
# tie, then the window rank of the score route), only while positive, and
# the first one that does not fit ends the allocation (a single multiplier).
# The result decides (n_fp, n_q); the windows are then assigned by score rank
# as in the score route.

RD_EQ = 1.0 - 2.0 ** -2            # distortion removed by E -> INT2, per unit weight
RD_QF = 2.0 ** -2 - 2.0 ** -16     # by INT2 -> FP


def rd_counts(S_desc, L: int, w: int, Hkv: int, d: int, beta: float):
    """(n_fp, n_q) of the rate-distortion allocation for one sequence; S_desc
    are the scores of the candidate windows other than the open one, in rank
    order (highest first)."""
    c_fp, c_q = window_costs(w, Hkv, d)
    Bt = budget_bytes(L, Hkv, d, beta)
    if Bt < c_fp:
        raise BudgetError(f"budget {Bt} B cannot hold the open window ({c_fp} B)")
    alpha = RD_EQ / c_q
    gamma = RD_QF / (c_fp - c_q)
    used, a, f, n = c_fp, 0, 0, len(S_desc)
    while True:
        eq = alpha * float(S_desc[a]) if a < n else -math.inf
        qf = gamma * float(S_desc[f]) if f < a else -math.inf
        if max(eq, qf) <= 0.0:
            break
        cost = c_q if eq >= qf else c_fp - c_q
        if used + cost > Bt:
            break
        used += cost
        if eq >= qf:
            a += 1
        else:
            f += 1
    return 1 + f, a - f


def route_rd(cache, scores_override=None):
    """A routing event by the rate-distortion allocation (scores as in route)."""
    if scores_override is not None:
        ov = np.asarray(scores_override, np.float64)
        cache.S = [ov[b, :cache.W].copy() for b in range(cache.B)]
    counts = []
    W = cache.W
    for b in range(cache.B):
        old = cache.tiers_now(b)
        S = cache.S[b]
        cand = [i for i in range(W) if old[i] != TIER_E]
        if not all(math.isfinite(float(S[i])) for i in cand):
            raise OracleError("non-finite score among routing candidates")
        forced = W - 1
        order = sorted(cand, key=lambda i: (i != forced, -float(S[i]), i))
        n_fp, n_q = rd_counts([S[i] for i in order[1:]], cache.L, cache.w, cache.Hkv, cache.d, cache.beta)
        new = np.array(old, np.uint8)
        for r, i in enumerate(order):
            new[i] = TIER_FP if r < n_fp else (TIER_Q if r < n_fp + n_q else TIER_E)
        cache.apply_tiers(b, new)
        counts.append(transition_counts(old, cache.tiers_now(b)))
    cache.last_counts = np.stack(counts)


# ---- rate-distortion routing over all widths {0, 2, 4, 8, 16} (an option) ----
#
# The same allocation with RDKV's full width set. A window's options form a
# chain of widths: 0 -> 2 -> 4 -> 8 -> 16 for a window never quantised, and
# 0 -> b -> 16 for one whose ledger entry has width b (the write-once ledger
# fixes the width at the first quantisation). Each step of a chain is an
# upgrade removing (2^-a - 2^-b) w of distortion for cost(b) - cost(a) bytes;
# its gain per byte is k_step * w with k_step = (2^-a - 2^-b) / (cost(b) -
# cost(a)) (one float64 product per upgrade). Along every chain k_step falls,
# so taking the upgrades of all windows in order of gain per byte, highest
# first (a lower step first on a tie, then the window rank), while positive,
# until the first that does not fit, takes each chain's steps in order: the
# Lagrangian solution of the multiple-choice knapsack.

def width_cost(w: int, Hkv: int, d: int, bits: int) -> int:
    """Bytes of one window at a width: 0 evicted, 16 bf16, else codes + fp16 meta."""
    if bits == 0:
        return 0
    if bits == 16:
        return w * Hkv * d * 4
    return w * Hkv * 2 * (d * bits // 8 + 4 * (d // GROUP))


def rd_mixed_widths(S_ranked, chains, L: int, w: int, Hkv: int, d: int, beta: float):
    """Widths of the candidates other than the open window, given in rank
    order with their chains (lists of widths starting at 0)."""
    c_fp = width_cost(w, Hkv, d, 16)
    Bt = budget_bytes(L, Hkv, d, beta)
    if Bt < c_fp:
        raise BudgetError(f"budget {Bt} B cannot hold the open window ({c_fp} B)")
    ups = []
    for r, (s, ch) in enumerate(zip(S_ranked, chains)):
        for i in range(len(ch) - 1):
            a, b = ch[i], ch[i + 1]
            cost = width_cost(w, Hkv, d, b) - width_cost(w, Hkv, d, a)
            k = (2.0 ** -a - 2.0 ** -b) / cost
            ups.append((k * float(s), i, r, cost))
    ups.sort(key=lambda u: (-u[0], u[1], u[2]))
    used, steps = c_fp, [0] * len(chains)
    for gain, i, r, cost in ups:
        if gain <= 0.0 or used + cost > Bt:
            break
        assert steps[r] == i, "a chain's steps come in order"
        used += cost
        steps[r] += 1
    return [ch[st] for ch, st in zip(chains, steps)]


def route_rd_mixed(cache, scores_override=None, max_bits=8):
    """A routing event by the rate-distortion allocation over widths
    {0, 2, 4, 8, 16} (those up to max_bits, and 16); windows keep the width of
    an existing ledger entry."""
    if scores_override is not None:
        ov = np.asarray(scores_override, np.float64)
        cache.S = [ov[b, :cache.W].copy() for b in range(cache.B)]
    counts = []
    W = cache.W
    for b in range(cache.B):
        old = cache.tiers_now(b)
        S = cache.S[b]
        cand = [i for i in range(W) if old[i] != TIER_E]
        if not all(math.isfinite(float(S[i])) for i in cand):
            raise OracleError("non-finite score among routing candidates")
        forced = W - 1
        order = sorted(cand, key=lambda i: (i != forced, -float(S[i]), i))
        rest = order[1:]
        free = [0] + [x for x in (2, 4, 8) if x <= max_bits] + [16]
        chains = [free if cache.win[b][i].ledger is None else [0, cache.win[b][i].ledger_bits, 16]
                  for i in rest]
        widths = rd_mixed_widths([S[i] for i in rest], chains, cache.L, cache.w, cache.Hkv, cache.d, cache.beta)
        new = np.array(old, np.uint8)
        if order:   # the first-ranked candidate (the open window) stays full precision, as in route_rd
            new[order[0]] = TIER_FP
        for i, bits in zip(rest, widths):
            new[i] = TIER_OF_BITS[bits]
        cache.apply_tiers(b, new)
        counts.append(transition_counts(old, cache.tiers_now(b)))
    cache.last_counts = np.stack(counts)


# ---- a positional router (an option) ----------------------------------------
#
# "Technische Samenvatting: LogQuant", Methodologie 1-2: high-attention
# positions thin out logarithmically with the distance to the current token,
# so LogQuant keeps the most recent tokens at full precision and, further
# back, tokens at a density that halves from region to region; the rest are
# 2-bit. The summary's numbers are garbled ("2W" and "3W" recent tokens), so
# at window granularity the reading is: the R most recent windows are dense;
# before them, region l = 1, 2, ... covers ages [R 2^(l-1), R 2^l) (age 0 is
# the open window) and first contributes the windows at spacing 2^l, then, in
# later rounds, the ones at half that spacing, and so on. A window's rank is
# (round, region, age), lowest first, so every top-k set is log-spaced and
# each includes the smaller ones. The budget counts and the evict / demote /
# promote moves are the score-based route's.

def logsparse_rank(age: int, recent: int):
    """(round, region, age) of a window `age` windows before the open one."""
    if age < recent:
        return (0, 0, age)
    region = 1
    while age >= recent << region:
        region += 1
    m = age - (recent << (region - 1))
    tz = region if m == 0 else min(region, (m & -m).bit_length() - 1)
    return (1 + region - tz, region, age)


def route_logsparse(cache, recent: int = 2):
    """A routing event of every sequence by log-sparse position instead of
    score: the windows' ranks replace the scores in route_tiers (the scores
    themselves are left as they are)."""
    counts = []
    W = cache.W
    order = sorted(range(W), key=lambda i: logsparse_rank(W - 1 - i, recent))
    pseudo = np.zeros(W)
    for r, i in enumerate(order):
        pseudo[i] = -float(r)    # higher = earlier in the order
    for b in range(cache.B):
        old = cache.tiers_now(b)
        new = route_tiers(pseudo, old, cache.L, cache.w, cache.Hkv, cache.d, cache.beta, cache.rho)
        cache.apply_tiers(b, new)
        counts.append(transition_counts(old, cache.tiers_now(b)))
    cache.last_counts = np.stack(counts)


# ---- one budget across layers and KV heads (an option) ------------------------
#
# "Technische Samenvatting: DBTrimKV", section 3 (global budget): instead of a
# budget per layer or head, one budget M_global for the whole cache, every
# cached entry ranked globally by one utility score and the top ones kept.
# Here the utility is the cumulative attention score: every layer spreads one
# unit of mass per query head per decode step over its windows, so the
# layers' scores share a scale without learned gates. The QEvict rule is
# applied unchanged with the candidate set, the budget and the forced windows
# widened to all layers (and, with per-head units, all KV heads) of a
# sequence:
#   budget   B_g = floor(beta * sum over the layers and units of L * Hkv * d * 4)
#   forced   the last window of every unit of every layer (full precision)
#   counts   n_fp = min(C, max(n_forced, floor(rho * B_g / c_fp))),
#            n_q  = min(C - n_fp, floor((B_g - n_fp * c_fp) / c_q))
#   ranking  forced first, then score descending, then (layer, unit, window)
#            ascending; top n_fp full precision, next n_q INT2, rest evicted.

def route_global(layers, hs=1, scores_override=None):
    """One routing event over several layers under one byte budget per
    sequence. `layers`: OracleCache per layer with the same units and window;
    `hs`: units per sequence (1, or Hkv with per-head units); scores_override:
    optional list (per layer) of [units][W] arrays replacing the scores.
    Moves every layer's tiers (evict, demote, promote per unit) and sets each
    layer's last_counts; raises BudgetError if the forced windows do not fit."""
    if scores_override is not None:
        for c, ov in zip(layers, scores_override):
            ov = np.asarray(ov, np.float64)
            c.S = [ov[u, :c.W].copy() for u in range(c.B)]
    first = layers[0]
    U, w, d = first.B, first.w, first.d
    c_fp, c_q = window_costs(w, first.Hkv, d)
    new = [c.tiers().copy() for c in layers]
    for b in range(U // hs):
        units = range(b * hs, (b + 1) * hs)
        F = sum(c.L * c.Hkv * d * 4 for c in layers for _ in units)
        Bg = int(math.floor(first.beta * F))
        forced, cand = [], []
        for li, c in enumerate(layers):
            for j, u in enumerate(units):
                W = c.W
                for wi in range(W):
                    if c.win[u][wi].tier == TIER_E:
                        continue
                    s = float(c.S[u][wi])
                    if not math.isfinite(s):
                        raise OracleError("non-finite score among routing candidates")
                    (forced if wi == W - 1 else cand).append((li, j, wi, s))
        if not forced and not cand:
            continue
        if len(forced) * c_fp > Bg:
            raise BudgetError(f"budget {Bg} B cannot hold the {len(forced)} open windows")
        C = len(forced) + len(cand)
        n_fp = min(C, max(len(forced), fp_budget_windows(Bg, c_fp, first.rho)))
        n_q = min(C - n_fp, (Bg - n_fp * c_fp) // c_q)
        order = sorted(forced, key=lambda e: e[:3]) + sorted(cand, key=lambda e: (-e[3], e[0], e[1], e[2]))
        for r, (li, j, wi, _) in enumerate(order):
            new[li][b * hs + j, wi] = TIER_FP if r < n_fp else (TIER_Q if r < n_fp + n_q else TIER_E)
    for li, c in enumerate(layers):
        counts = []
        for u in range(U):
            old = c.tiers_now(u)
            c.apply_tiers(u, new[li][u])
            counts.append(transition_counts(old, c.tiers_now(u)))
        c.last_counts = np.stack(counts)



# ---- the K-channel half of the rate-distortion allocation (an option) -------
#
# "Technische Samenvatting: RDKV", 2.1: the distortion weight of a K-cache
# channel c is the spectral norm of the logit change when the channel is set
# to zero, w_c = (1/sqrt(d)) ||Q[:, c]||_2 ||K[:, c]||_2. 2.2: the weights are
# computed once after the prefill (Fase 1); the channels then take widths by
# the same Lagrangian knapsack, over the tokens Fase 2 kept (Fase 3), so one
# token's K and V can have different widths. 2.3: the K rows of the packed old
# stream (Zone A) carry widths {2, 4, 8}.
#
# Readings (the library follows the same ones):
# * Q is the set of query vectors the caller observed over the prefill; the G
#   query heads of a KV head pool their columns ([positions x G] rows).
# * Units are the quantiser's groups of 32 channels per KV head: channels of a
#   group share a scale, so they share a width; a group's weight is the sum of
#   its 32 channel weights (float32 weights added in channel order in
#   float64). The widths are {0, 2, 4, 8}: 0 drops the group's channels from
#   the logits, 16-bit K belongs to full-precision windows (Zone B/C).
# * Every group keeps its fp16 scale and minimum (zero for a dropped group), so
#   a group costs 4 b + 4 bytes per token at width b.
# * The K budget is what the K halves of the windows Fase 2 quantised occupy at
#   their widths; the channel allocation redistributes it over the groups of
#   all KV heads of the sequence: from all groups at 0, steps a -> b along
#   0 -> 2 -> 4 -> 8 with gain (2^-a - 2^-b) W_g per byte are taken by gain,
#   highest first (a lower step, then the lower unit (KV head, group) on a
#   tie), while positive, until the first that does not fit, as in A31.
# * The allocation runs with the layer's first quantisation: the K widths are
#   then fixed for the sequence (the ledger is written once), and the layer
#   takes no further routing events or listed moves.

K_WIDTHS = (0, 2, 4, 8)


def k_channel_weights(q_obs, k_full, Hkv: int):
    """RDKV 2.1's K-channel weights, float64 [B][Hkv][d].

    q_obs: [B][n_q][Hq][d] observed queries; k_full: [B][n][Hkv][d] the keys."""
    q = np.asarray(q_obs, np.float64)
    k = np.asarray(k_full, np.float64)
    B, nq, Hq, d = q.shape
    G = Hq // Hkv
    qg = q.reshape(B, nq, Hkv, G, d)
    qn = np.sqrt((qg * qg).sum(axis=(1, 3)))            # [B][Hkv][d]
    kn = np.sqrt((k * k).sum(axis=1))                   # [B][Hkv][d]
    return qn * kn / math.sqrt(d)


def k_group_cost(bits: int) -> int:
    """Bytes one token spends on one 32-channel K group at a width."""
    return GROUP * bits // 8 + 4


def k_channel_widths(weights32, n_tok: int, budget: int):
    """Widths [Hkv][4] of one sequence's K groups (Fase 3), given the float32
    channel weights [Hkv][d], the tokens of the quantised windows and the K
    budget in bytes."""
    wts = np.asarray(weights32, np.float32)
    Hkv, d = wts.shape
    ng = d // GROUP
    units = [(h, g) for h in range(Hkv) for g in range(ng)]
    Wg = [sum(float(x) for x in wts[h, g * GROUP:(g + 1) * GROUP]) for h, g in units]
    widths = [0] * len(units)
    if n_tok <= 0:
        return np.zeros((Hkv, ng), np.int64)
    used = n_tok * len(units) * k_group_cost(0)
    ups = []
    for u, W in enumerate(Wg):
        for i in range(len(K_WIDTHS) - 1):
            a, b = K_WIDTHS[i], K_WIDTHS[i + 1]
            cost = n_tok * (k_group_cost(b) - k_group_cost(a))
            kk = (2.0 ** -a - 2.0 ** -b) / cost
            ups.append((kk * W, i, u, cost))
    ups.sort(key=lambda e: (-e[0], e[1], e[2]))
    steps = [0] * len(units)
    for gain, i, u, cost in ups:
        if gain <= 0.0 or used + cost > budget:
            break
        assert steps[u] == i, "a group's steps come in order"
        used += cost
        steps[u] += 1
    for u in range(len(units)):
        widths[u] = K_WIDTHS[steps[u]]
    return np.array(widths, np.int64).reshape(Hkv, ng)


def quantize_k_groups(x, kw):
    """K of one window ([Hkv][w][ng][32] bf16 values) with group g of KV head h
    at width kw[h][g]: codes, fp16 scale and minimum as quantize_groups gives
    them at that width; a group at width 0 has zero codes and meta."""
    x = np.asarray(x, np.float32)
    Hkv, w, ng, _ = x.shape
    codes = np.zeros(x.shape, np.uint8)
    s16 = np.zeros((Hkv, w, ng), np.float16)
    m16 = np.zeros((Hkv, w, ng), np.float16)
    bad = np.zeros((Hkv, w, ng), bool)
    for h in range(Hkv):
        for g in range(ng):
            bits = int(kw[h][g])
            if bits == 0:
                continue
            c, sc, mn, bd = quantize_groups(x[h, :, g], bits)
            codes[h, :, g], s16[h, :, g], m16[h, :, g], bad[h, :, g] = c, sc, mn, bd
    return codes, s16, m16, bad


def route_rd_kv(cache, weights32, scores_override=None, max_bits=8):
    """The rate-distortion route with the K-channel half: the window widths of
    route_rd_mixed (Fase 2), then the K group widths of each sequence
    (Fase 3, k_channel_widths) from the float32 channel weights [B][Hkv][d];
    the quantised windows' K groups take those widths, their V the window's.
    Needs a layer none of whose windows has been quantised."""
    if cache.kch is not None or any(win.ledger is not None for b in range(cache.B) for win in cache.win[b]):
        raise StateError("the K-channel widths are set with the layer's first quantisation")
    wts = np.asarray(weights32, np.float32)
    if scores_override is not None:
        ov = np.asarray(scores_override, np.float64)
        cache.S = [ov[b, :cache.W].copy() for b in range(cache.B)]
    W = cache.W
    plans = []
    for b in range(cache.B):
        old = cache.tiers_now(b)
        S = cache.S[b]
        cand = [i for i in range(W) if old[i] != TIER_E]
        if not all(math.isfinite(float(S[i])) for i in cand):
            raise OracleError("non-finite score among routing candidates")
        forced = W - 1
        order = sorted(cand, key=lambda i: (i != forced, -float(S[i]), i))
        rest = order[1:]
        free = [0] + [x for x in (2, 4, 8) if x <= max_bits] + [16]
        widths = rd_mixed_widths([S[i] for i in rest], [free] * len(rest), cache.L, cache.w, cache.Hkv,
                                 cache.d, cache.beta)
        new = np.array(old, np.uint8)
        if order:
            new[order[0]] = TIER_FP
        for i, bits in zip(rest, widths):
            new[i] = TIER_OF_BITS[bits]
        q_bits = [bits for bits in widths if bits in (2, 4, 8)]
        n_tok = len(q_bits) * cache.w
        k_budget = sum(width_cost(cache.w, cache.Hkv, cache.d, bits) // 2 for bits in q_bits)
        plans.append((old, new, k_channel_widths(wts[b], n_tok, k_budget)))
    cache.kch = np.stack([p[2] for p in plans])
    counts = []
    for b, (old, new, _) in enumerate(plans):
        cache.apply_tiers(b, new)
        counts.append(transition_counts(old, cache.tiers_now(b)))
    cache.last_counts = np.stack(counts)
    cache.kch_locked = True
