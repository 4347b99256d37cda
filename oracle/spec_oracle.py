"""fp64 CPU oracle for the speculative-sampling verify step, the draft/target
overlap statistics and the E2E-TV loss.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links
this module: it is used by ``tests/``, by ``__graft_entry__.smoke()`` and by
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``.  It shares no
code with the CUDA path.

Every function is a plain restatement of a definition printed on one of three
pages, cited by page title and section:

* "读 Qwen Bebop 与 DeepSeek DSpark：Speculative Decoding 正在从技巧变成系统工程"
  (cited below as *Bebop/DSpark blog*),
* "SpecOPD: Branch-Parallel On-Policy Distillation for Speculative Decoding"
  (cited as *SpecOPD summary*),
* "Speculative Decoding 与 MTP：先猜多个 token，再让大模型一次验完"
  (cited as *Speculative Decoding 与 MTP*).

Arithmetic is float64 throughout (bf16 / fp32 inputs are widened exactly).
The core routines (``overlap``, ``residual``, ``inverse_cdf``,
``verify_row_probs``) only use numpy operations that also work on object
arrays of ``fractions.Fraction``, so the tests can run them in exact rational
arithmetic.

Readings taken where the pages are silent or garbled (each is listed, with the
reason, in the design notes of the repository):

* accept iff ``u <= p(y)/q(y)`` with ``u`` in [0, 1);
* the residual is ``max(0, p - q)`` normalised by its own sum (the formula
  itself is lost on the page; the proof that follows it states the terms);
* inverse CDF in vocabulary order: the smallest ``v`` whose running sum
  exceeds ``u' * total``;
* one final uniform ``u'`` per row, used by the correction or by the bonus
  (exactly one of them happens);
* a rejection whose residual mass is exactly zero (possible only through
  rounding) samples from ``p`` instead and is reported;
* greedy ties go to the smallest index; the overlap at ``T == 0`` is the
  indicator ``[argmax p == argmax q]``;
* the E2E-TV loss is ``mean_b sum_j prod_{k<=j} alpha_{b,k}`` (to be
  maximised) and its gradient is taken with respect to the draft logits only,
  the target being a constant; the sub-gradient of ``min`` uses the strict
  indicator ``1[q_v < p_v]``.
* relaxed (lossy) acceptance: a draft is accepted when it ranks in the
  target's top-k (ties by smaller index) and its target log-probability lies
  within delta of the largest; the first rejection emits a draw from the
  full target distribution (no residual), the bonus stays as in the exact
  verify;
* a candidate tree's greedy verify walks from the prefix to the first child
  (in node order) whose token is the target argmax of the current slot, and
  emits that argmax where no child matches;
* top-k / top-p truncation ranks tokens by logit (ties by smaller index),
  applies top-k first, then keeps the shortest ranked prefix whose
  renormalised mass at temperature T reaches top_p; dropped logits become
  -inf, on the target and the draft alike.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
against closed forms, worked examples printed on the pages, exact rational
enumeration, chi-square tests and finite differences.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# Distance below which the oracle reports that a floating-point decision sits
# on a boundary (|u - p/q| or |C_v/Z - u'|).  Integer outputs of another
# implementation are compared with the oracle's only where no flag is raised.
NEAR_TIE = 1e-6


# ---------------------------------------------------------------------------
# Distributions
# ---------------------------------------------------------------------------

def softmax_t(z, temperature):
    """Temperature softmax of one logit row.

    Target and draft distributions p(y), q(y) -- Bebop/DSpark blog, section
    "用公式看：到底什么叫“猜得值”" (definitions of p and q); both sides use the
    same temperature -- Speculative Decoding 与 MTP, section 4.
    """
    z = np.asarray(z, dtype=np.float64)
    t = float(temperature)
    if not t > 0.0:
        raise ValueError("softmax_t needs a positive temperature")
    a = (z - np.max(z)) / t
    e = np.exp(a)
    return e / np.sum(e)


# ---------------------------------------------------------------------------
# Top-k / top-p truncation, applied the same way to target and draft logits
# ---------------------------------------------------------------------------

# Distance (in probability mass) below which a top-p cut is reported as a
# near tie: another implementation's rounding may move the cut by one token.
NEAR_TRUNC = 1e-5


def truncate_logits(z, temperature, top_k=0, top_p=1.0):
    """Top-k, then top-p truncation of one logit row, as sampling applies it.

    Speculative Decoding 与 MTP, section 4: p and q must both be computed after
    the agreed temperature and top-k / top-p transforms; section 23: a mask
    applied to one side only breaks correctness.  The pages give no formula;
    the transform taken is the common one:

    * tokens are ranked by logit, larger first, ties by smaller index;
    * top-k (0 < top_k < V) keeps the first top_k tokens of that ranking;
    * top-p (top_p < 1) renormalises softmax(z / T) over the kept tokens and
      keeps, in ranking order, every token whose preceding mass is below
      top_p (the shortest prefix reaching top_p);
    * dropped tokens get logit -inf; kept tokens keep their logit.

    Returns ``(z_out, near)``; ``near`` reports a top-p cut whose preceding
    mass lies within NEAR_TRUNC of top_p on either side of the boundary.
    """
    z = np.asarray(z, dtype=np.float64)
    V = z.shape[0]
    order = np.lexsort((np.arange(V), -z))  # logit descending, then index ascending
    keep = np.ones(V, dtype=bool)
    if 0 < top_k < V:
        keep[:] = False
        keep[order[:top_k]] = True
    near = False
    if top_p < 1.0:
        ranked = order[keep[order]]  # kept tokens in ranking order
        p = softmax_t(z[ranked], temperature)
        before = np.concatenate(([0.0], np.cumsum(p)[:-1]))
        sel = before < top_p
        n = int(sel.sum())
        near = bool(abs(before[n - 1] - top_p) < NEAR_TRUNC or
                    (n < before.size and abs(before[n] - top_p) < NEAR_TRUNC))
        keep[:] = False
        keep[ranked[:n]] = True
    return np.where(keep, z, -np.inf), near


def overlap(p, q):
    """alpha = sum_v min(p(v), q(v)).

    The expected single-step acceptance rate of rejection sampling equals the
    overlap mass -- Bebop/DSpark blog, section "用公式看", equation for
    alpha_RS; SpecOPD summary, "验收长度与 E2E-TV 目标".
    """
    return np.sum(np.minimum(p, q))


def tv_distance(p, q):
    """d_TV(p, q) = 1/2 sum_v |p(v) - q(v)|, computed independently of
    ``overlap`` -- Bebop/DSpark blog, section "用公式看", definition of d_TV."""
    return np.sum(np.abs(p - q)) / 2


def residual(p, q):
    """Unnormalised residual max(0, p - q).

    The correction after a rejection draws from the target's mass left over
    by the drafter -- Speculative Decoding 与 MTP, section 3 (the formula is
    lost; its proof names the rejected-path term max(0, p(v) - q(v))).
    """
    return np.maximum(p - q, 0)


def inverse_cdf(w, u):
    """Draw from the (unnormalised, non-negative) weights ``w`` with one
    uniform ``u`` in [0, 1): the smallest index v with
    sum_{i<=v} w_i > u * sum_i w_i (vocabulary order).

    Returns ``(v, near)`` where ``near`` reports that ``u`` lies within
    ``NEAR_TIE`` of the CDF boundary below or above the chosen index.
    """
    c = np.cumsum(w)
    total = c[-1]
    if not total > 0:
        raise ValueError("inverse_cdf needs positive total mass")
    thr = u * total
    above = np.nonzero(c > thr)[0]
    if above.size:
        v = int(above[0])
    else:  # rounding can leave u*total == total; take the last positive weight
        v = int(np.nonzero(w > 0)[0][-1])
    hi = c[v] / total
    lo = c[v - 1] / total if v > 0 else 0 * total
    near = bool(abs(hi - u) < NEAR_TIE or abs(u - lo) < NEAR_TIE)
    return v, near


def argmax_first(z):
    """Greedy choice with ties broken towards the smallest index."""
    return int(np.argmax(np.asarray(z)))


# ---------------------------------------------------------------------------
# Acceptance length
# ---------------------------------------------------------------------------

def prefix_survival(alpha):
    """a_j = P(tau >= j) = prod_{k<=j} alpha_k for j = 1..K.

    Bebop/DSpark blog, section "用公式看" (P(tau >= j)) and section
    "DSpark 的第二块拼图" (a_j = prod c_i).
    """
    out = []
    acc = 1
    for a in alpha:
        acc = acc * a
        out.append(acc)
    return out


def expected_accepted(alpha):
    """E[tau] = sum_{j=1..K} prod_{k<=j} alpha_k (no bonus token).

    Bebop/DSpark blog, section "用公式看", equation for E[tau].
    """
    s = 0
    for a in prefix_survival(alpha):
        s = s + a
    return s


def expected_emitted(alpha):
    """Expected tokens emitted by one cycle: the accepted drafts plus the one
    correction or bonus token, 1 + E[tau] -- Speculative Decoding 与 MTP,
    section 6 (worked example 1+0.8+0.64+0.512+0.4096) and section 7."""
    return 1 + expected_accepted(alpha)


# ---------------------------------------------------------------------------
# Verify
# ---------------------------------------------------------------------------

@dataclass
class RowResult:
    tokens: list          # K+1 ints, -1 after the last emitted token
    n_accepted: int       # number of accepted drafts, 0..K
    alpha: list           # K overlaps
    tv: list              # K total-variation distances
    accept_near: bool     # some evaluated |u_k - p/q| < NEAR_TIE
    cdf_near: bool        # the correction / bonus draw sits on a CDF boundary
    residual_empty: bool  # rejection with zero residual mass (rounding only)


def accept_and_correct(p, q, draft, u_accept, u_final):
    """The sampling decisions of one row, given the distributions.

    p: K+1 target distributions (p_1..p_K and the bonus distribution
       p_{K+1}); q: K draft distributions; draft: K drafted token ids;
    u_accept: K uniforms; u_final: one uniform for the correction / bonus.

    Steps, in the order of Speculative Decoding 与 MTP, sections 2 and 3:
    accept draft k with probability min(1, p_k(y)/q_k(y)), in prefix order;
    the first rejection ends the block and emits a token drawn from the
    normalised residual max(0, p_k - q_k); if every draft is accepted, the
    bonus token is drawn from p_{K+1}.

    Returns (tokens, n_accepted, accept_near, cdf_near, residual_empty).
    """
    K = len(q)
    tokens = [-1] * (K + 1)
    accept_near = False
    cdf_near = False
    residual_empty = False
    n = K
    for k in range(K):
        y = int(draft[k])
        pk, qk = p[k][y], q[k][y]
        u = u_accept[k]
        if qk > 0:
            r = pk / qk
            if abs(u - r) < NEAR_TIE:
                accept_near = True
            accepted = u <= r
        else:  # q(y) == 0: the ratio is +inf, always accept
            accepted = True
        if accepted:
            tokens[k] = y
            continue
        rho = residual(p[k], q[k])
        if rho.sum() > 0:
            v, cdf_near = inverse_cdf(rho, u_final)
        else:
            residual_empty = True
            v, cdf_near = inverse_cdf(p[k], u_final)
        tokens[k] = v
        n = k
        break
    else:
        v, cdf_near = inverse_cdf(p[K], u_final)
        tokens[K] = v
    return tokens, n, accept_near, cdf_near, residual_empty


def verify_row_probs(p, q, draft, u_accept, u_final):
    """One row of the verify step: the sampling decisions of
    ``accept_and_correct`` plus the per-position overlap and d_TV."""
    K = len(q)
    alpha = [overlap(p[k], q[k]) for k in range(K)]
    tv = [tv_distance(p[k], q[k]) for k in range(K)]
    tokens, n, a_near, c_near, empty = accept_and_correct(p, q, draft, u_accept, u_final)
    return RowResult(tokens, n, alpha, tv, a_near, c_near, empty)


def verify_row_greedy(zt, zd, draft):
    """Greedy (T == 0) verify of one row: compare each draft with the target
    argmax; at the first mismatch emit the target argmax, else emit the argmax
    of the bonus position -- Speculative Decoding 与 MTP, section 4.

    The overlap is the one-hot limit [argmax p == argmax q]; zd may be None
    when the overlap is not wanted.
    """
    K = len(draft)
    tokens = [-1] * (K + 1)
    n = K
    for k in range(K):
        a = argmax_first(zt[k])
        if int(draft[k]) == a:
            tokens[k] = a
            continue
        tokens[k] = a
        n = k
        break
    else:
        tokens[K] = argmax_first(zt[K])
    if zd is None:
        alpha = [float("nan")] * K
    else:
        alpha = [1.0 if argmax_first(zt[k]) == argmax_first(zd[k]) else 0.0
                 for k in range(K)]
    tv = [1.0 - a for a in alpha]
    return RowResult(tokens, n, alpha, tv, False, False, False)


@dataclass
class VerifyResult:
    tokens: np.ndarray          # int64 [B, K+1]
    n_accepted: np.ndarray      # int64 [B]
    alpha: np.ndarray           # float64 [B, K]
    tv: np.ndarray              # float64 [B, K]
    prefix_survival: np.ndarray  # float64 [B, K]
    accept_near: np.ndarray     # bool [B]
    cdf_near: np.ndarray        # bool [B]
    residual_empty: np.ndarray  # bool [B]

    @property
    def flagged(self):
        return self.accept_near | self.cdf_near


def verify(target_logits, draft_logits, draft_tokens, u_accept, u_final,
           temperature, rows=None):
    """Batched verify: target_logits [B, K+1, V], draft_logits [B, K, V],
    draft_tokens [B, K], u_accept [B, K], u_final [B]; temperature >= 0
    (0 selects greedy).  ``rows`` restricts the work to a subset of batch
    rows (outputs then have len(rows) rows)."""
    zt = np.asarray(target_logits)
    zd = None if draft_logits is None else np.asarray(draft_logits)
    B, K1, V = zt.shape
    K = K1 - 1
    rows = range(B) if rows is None else list(rows)
    R = len(rows)
    tokens = np.full((R, K + 1), -1, dtype=np.int64)
    n_acc = np.zeros(R, dtype=np.int64)
    alpha = np.zeros((R, K))
    tv = np.zeros((R, K))
    surv = np.zeros((R, K))
    a_near = np.zeros(R, dtype=bool)
    c_near = np.zeros(R, dtype=bool)
    r_empty = np.zeros(R, dtype=bool)
    t = float(temperature)
    for i, b in enumerate(rows):
        if t == 0.0:
            res = verify_row_greedy(zt[b].astype(np.float64),
                                    None if zd is None else zd[b].astype(np.float64),
                                    draft_tokens[b])
        else:
            p = [softmax_t(zt[b, k], t) for k in range(K + 1)]
            q = [softmax_t(zd[b, k], t) for k in range(K)]
            res = verify_row_probs(p, q, draft_tokens[b], u_accept[b].astype(np.float64),
                                   float(u_final[b]))
        tokens[i] = res.tokens
        n_acc[i] = res.n_accepted
        alpha[i] = res.alpha
        tv[i] = res.tv
        surv[i] = prefix_survival(res.alpha) if K else []
        a_near[i] = res.accept_near
        c_near[i] = res.cdf_near
        r_empty[i] = res.residual_empty
    return VerifyResult(tokens, n_acc, alpha, tv, surv, a_near, c_near, r_empty)


# ---------------------------------------------------------------------------
# Tree-shaped candidates: the tree attention mask and the greedy verify
# ---------------------------------------------------------------------------

def tree_mask(parent):
    """Tree attention mask of a candidate tree given by its parent map
    (parent[i] < i, -1 for a node hung on the committed prefix): M[u, v] = 1
    iff v is u or a strict ancestor of u.  SpecOPD summary, section "树注意力
    (Tree Attention)": each node sees only its ancestors and itself, so one
    batched pass scores every node without leaking sibling branches.  Also
    returns each node's depth (0 for a node hung on the prefix), its position
    in the sequence it belongs to."""
    parent = [int(x) for x in parent]
    N = len(parent)
    M = np.zeros((N, N), dtype=bool)
    depth = np.zeros(N, dtype=np.int64)
    for u in range(N):
        v = u
        while v >= 0:
            M[u, v] = True
            v = parent[v]
        depth[u] = int(M[u].sum()) - 1
    return M, depth


@dataclass
class TreeResult:
    path: np.ndarray        # int64 [B, N]: accepted nodes, root side first, -1 after
    tokens: np.ndarray      # int64 [B, N + 1]: their tokens, then the target's token, -1 after
    n_accepted: np.ndarray  # int64 [B]


def tree_verify_greedy(target_logits, parent, node_tokens):
    """Greedy (T == 0) verify of a candidate tree, committing one path.

    Speculative Decoding 与 MTP, section 4 (greedy: a candidate is kept when
    it equals the target argmax; at the first mismatch the target's token is
    used) and section 11 (a tree of candidates commits a single path).

    target_logits [B, N + 1, V]: slot 0 holds the target's logits after the
    committed prefix, slot i + 1 those after candidate node i (one batched
    target pass over the tree with ``tree_mask``).  parent [B, N] with
    parent[b, i] < i (-1: hung on the prefix); node_tokens [B, N].  From the
    prefix, the walk moves to the first child (in node order) whose token is
    the argmax (smallest index on ties) of the current slot; where no child
    matches it emits that argmax and stops."""
    zt = np.asarray(target_logits)
    B, N1, V = zt.shape
    N = N1 - 1
    parent = np.asarray(parent)
    toks = np.asarray(node_tokens)
    path = np.full((B, N), -1, dtype=np.int64)
    out = np.full((B, N + 1), -1, dtype=np.int64)
    n_acc = np.zeros(B, dtype=np.int64)
    for b in range(B):
        cur, n = -1, 0
        while True:
            a = argmax_first(zt[b, cur + 1])
            nxt = next((c for c in range(N) if int(parent[b, c]) == cur and int(toks[b, c]) == a), None)
            if nxt is None:
                out[b, n] = a
                break
            path[b, n] = nxt
            out[b, n] = a
            n += 1
            cur = nxt
        n_acc[b] = n
    return TreeResult(path, out, n_acc)


# ---------------------------------------------------------------------------
# Relaxed (lossy) acceptance
# ---------------------------------------------------------------------------

def relaxed_accept(z, y, temperature, top_k, delta):
    """Relaxed acceptance of drafted token y against target logits z: y must
    rank among the target's top_k tokens (by logit, ties to the smaller
    index; top_k <= 0: no such condition) and its target log-probability may
    fall at most delta below the target's largest (delta = inf: no such
    condition).  Speculative Decoding 与 MTP, section 4: accepting a candidate
    that lies in the target's top-k, or whose logprob is close, raises the
    acceptance rate but no longer preserves the target distribution (the
    relaxed_topk / relaxed_delta switches it cites); such runs are lossy.

    Returns (accepted, near): near reports |gap + delta| < NEAR_TIE, gap the
    log-probability difference."""
    z = np.asarray(z, dtype=np.float64)
    V = z.shape[0]
    if not 0 <= y < V:
        return False, False
    zy = z[y]
    rank = int(np.sum(z > zy) + np.sum(z[:y] == zy))
    gap = (zy - np.max(z)) / float(temperature)
    ok_k = top_k <= 0 or rank < top_k
    ok_d = not np.isfinite(delta) or gap >= -delta
    near = bool(np.isfinite(delta) and abs(gap + delta) < NEAR_TIE)
    return bool(ok_k and ok_d), near


def verify_relaxed(target_logits, draft_logits, draft_tokens, u_final, temperature, top_k, delta,
                   rows=None):
    """Verify with relaxed acceptance (LOSSY): drafted tokens are accepted in
    prefix order while ``relaxed_accept`` holds; the first rejected position
    emits a draw from the full target distribution p_k with u' (a residual has
    no meaning once acceptance no longer follows min(1, p/q)), and a block with
    every draft accepted emits the bonus draw from p_{K+1}, as in the exact
    verify.  Overlaps are reported as for the exact verify when draft logits
    are given."""
    zt = np.asarray(target_logits)
    zd = None if draft_logits is None else np.asarray(draft_logits)
    B, K1, V = zt.shape
    K = K1 - 1
    rows = range(B) if rows is None else list(rows)
    R = len(rows)
    tokens = np.full((R, K + 1), -1, dtype=np.int64)
    n_acc = np.zeros(R, dtype=np.int64)
    alpha = np.zeros((R, K))
    tv = np.zeros((R, K))
    surv = np.zeros((R, K))
    a_near = np.zeros(R, dtype=bool)
    c_near = np.zeros(R, dtype=bool)
    t = float(temperature)
    for i, b in enumerate(rows):
        p = [softmax_t(zt[b, k], t) for k in range(K + 1)]
        if zd is not None:
            q = [softmax_t(zd[b, k], t) for k in range(K)]
            alpha[i] = [overlap(p[k], q[k]) for k in range(K)]
            tv[i] = [tv_distance(p[k], q[k]) for k in range(K)]
            surv[i] = prefix_survival(alpha[i]) if K else []
        n = K
        for k in range(K):
            y = int(draft_tokens[b][k])
            acc, near = relaxed_accept(zt[b, k], y, t, top_k, delta)
            a_near[i] |= near
            if acc:
                tokens[i, k] = y
                continue
            v, c_near[i] = inverse_cdf(p[k], float(u_final[b]))
            tokens[i, k] = v
            n = k
            break
        else:
            v, c_near[i] = inverse_cdf(p[K], float(u_final[b]))
            tokens[i, K] = v
        n_acc[i] = n
    return VerifyResult(tokens, n_acc, alpha, tv, surv, a_near, c_near, np.zeros(R, dtype=bool))


# ---------------------------------------------------------------------------
# Overlap statistics
# ---------------------------------------------------------------------------

@dataclass
class OverlapResult:
    alpha: np.ndarray             # [B, K]
    tv: np.ndarray                # [B, K]
    prefix_survival: np.ndarray   # [B, K]
    expected_accepted: np.ndarray  # [B]


def overlap_stats(target_logits, draft_logits, temperature, rows=None):
    """Per-position overlap alpha_k, d_TV, prefix survival prod_{k<=j} alpha_k
    and E[tau] for logits [B, K, V] (both sides) -- Bebop/DSpark blog, section
    "用公式看" and section "DSpark 的第二块拼图" (soft label c*_k = 1 - d_TV)."""
    zt = np.asarray(target_logits)
    zd = np.asarray(draft_logits)
    B, K, V = zt.shape
    rows = range(B) if rows is None else list(rows)
    R = len(rows)
    alpha = np.zeros((R, K))
    tv = np.zeros((R, K))
    t = float(temperature)
    for i, b in enumerate(rows):
        for k in range(K):
            if t == 0.0:
                a = 1.0 if argmax_first(zt[b, k]) == argmax_first(zd[b, k]) else 0.0
                alpha[i, k], tv[i, k] = a, 1.0 - a
            else:
                p = softmax_t(zt[b, k], t)
                q = softmax_t(zd[b, k], t)
                alpha[i, k] = overlap(p, q)
                tv[i, k] = tv_distance(p, q)
    surv = np.array([prefix_survival(alpha[i]) for i in range(R)]).reshape(R, K)
    exp_acc = surv.sum(axis=1)
    return OverlapResult(alpha, tv, surv, exp_acc)


# ---------------------------------------------------------------------------
# Entropy and acceptance diagnostics
# ---------------------------------------------------------------------------

def entropy(p):
    """H(p) = -sum_y p(y) log p(y) in nats, with 0 log 0 = 0.

    Bebop/DSpark blog, section "Qwen Bebop：RL 里的瓶颈不是 MTP 不会猜，而是
    策略熵在变" (the target policy's entropy that drives acceptance)."""
    p = np.asarray(p, dtype=np.float64)
    nz = p > 0
    return float(-np.sum(p[nz] * np.log(p[nz])))


def cross_entropy(p, q):
    """L_CE = -sum_y p(y) log q(y) in nats (terms with p(y) = 0 vanish).

    Bebop/DSpark blog, section "Bebop 的解法", equation for L_CE."""
    p = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    nz = p > 0
    return float(-np.sum(p[nz] * np.log(q[nz])))


def kl_divergence(p, q):
    """D_KL(p || q) = sum_y p(y) log(p(y) / q(y)) in nats (terms with p(y) = 0
    vanish) -- Bebop/DSpark blog, section "Bebop 的解法", equation for D_KL."""
    p = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    nz = p > 0
    return float(np.sum(p[nz] * np.log(p[nz] / q[nz])))


def alpha_target_only(p, q):
    """Single-step acceptance of target-only verification of a greedy draft:
    alpha_TO = p(y_hat) with y_hat = argmax_y q(y) (smallest index on ties).

    Bebop/DSpark blog, section "Qwen Bebop：RL 里的瓶颈...", equation for
    alpha_TO."""
    return float(np.asarray(p, dtype=np.float64)[argmax_first(q)])


@dataclass
class DiagResult:
    alpha: np.ndarray          # [B, K] sum min(p, q)
    entropy: np.ndarray        # [B, K] H(p), nats
    cross_entropy: np.ndarray  # [B, K] -sum p log q, nats
    kl: np.ndarray             # [B, K] D_KL(p || q), nats
    alpha_to: np.ndarray       # [B, K] p(argmax q)


def diagnostics(target_logits, draft_logits, temperature, rows=None):
    """Per-position overlap, target entropy, cross-entropy, KL divergence and
    target-only acceptance for logits [B, K, V] (both sides) at temperature
    T > 0; p and q are the temperature softmaxes of the two logit rows."""
    zt = np.asarray(target_logits)
    zd = np.asarray(draft_logits)
    B, K, V = zt.shape
    rows = range(B) if rows is None else list(rows)
    R = len(rows)
    out = [np.zeros((R, K)) for _ in range(5)]
    for i, b in enumerate(rows):
        for k in range(K):
            p = softmax_t(zt[b, k], temperature)
            q = softmax_t(zd[b, k], temperature)
            vals = (overlap(p, q), entropy(p), cross_entropy(p, q), kl_divergence(p, q),
                    alpha_target_only(p, q))
            for o, v in zip(out, vals):
                o[i, k] = v
    return DiagResult(*out)


# ---------------------------------------------------------------------------
# E2E-TV loss and its gradient with respect to the draft logits
# ---------------------------------------------------------------------------

def e2e_tv_loss(target_logits, draft_logits, temperature):
    """L = (1/B) sum_b sum_{j=1..K} prod_{k<=j} alpha_{b,k} with
    alpha_{b,k} = sum_v min(p_{b,k}(v), q_{b,k}(v)).

    Bebop/DSpark blog, section "Bebop 的解法", equation for E[tau] in terms of
    1 - d_TV; SpecOPD summary, "方法步骤详情" step (6) (prefix products of the
    per-position overlap).  Returns (L, alpha [B, K])."""
    zt = np.asarray(target_logits, dtype=np.float64)
    zd = np.asarray(draft_logits, dtype=np.float64)
    B, K, V = zt.shape
    alpha = np.zeros((B, K))
    for b in range(B):
        for k in range(K):
            alpha[b, k] = overlap(softmax_t(zt[b, k], temperature),
                                  softmax_t(zd[b, k], temperature))
    per_row = np.array([expected_accepted(alpha[b]) for b in range(B)])
    return float(per_row.sum() / B) if B else 0.0, alpha


def e2e_tv_grad(target_logits, draft_logits, temperature, grad_scale=1.0, rows=None):
    """Gradient of ``grad_scale * L`` with respect to the draft logits
    [B, K, V]; target and sampling are constants (SpecOPD summary,
    "方法步骤详情" step (6): only the draft probabilities are differentiated).

    Chain rule, written out:
      dL/dalpha_k = (1/B) * prod_{i<k} alpha_i * (1 + alpha_{k+1}
                    + alpha_{k+1} alpha_{k+2} + ...),
      dalpha_k/dz_v = (q_v / T) * (1[q_v < p_v] - S_k),
      S_k = sum_{u : q_u < p_u} q_u.
    Returns (grad [R, K, V], ambiguous [R, K, V]) where ``ambiguous`` marks
    elements whose indicator 1[q_v < p_v] lies within NEAR_TIE (relative) of
    flipping.  ``rows`` restricts the output to some batch rows (B in the
    1/B factor is still the full batch size).
    """
    zt = np.asarray(target_logits)
    zd = np.asarray(draft_logits)
    B, K, V = zt.shape
    t = float(temperature)
    rows = range(B) if rows is None else list(rows)
    R = len(rows)
    grad = np.zeros((R, K, V))
    amb = np.zeros((R, K, V), dtype=bool)
    for i, b in enumerate(rows):
        p = [softmax_t(zt[b, k], t) for k in range(K)]
        q = [softmax_t(zd[b, k], t) for k in range(K)]
        alpha = [overlap(p[k], q[k]) for k in range(K)]
        for k in range(K):
            before = 1.0
            for j in range(k):
                before *= alpha[j]
            after = 0.0
            chain = 1.0
            for j in range(k + 1, K):
                chain *= alpha[j]
                after += chain
            dl_dalpha = grad_scale * before * (1.0 + after) / B
            ind = (q[k] < p[k]).astype(np.float64)
            s_k = np.sum(q[k] * ind)
            grad[i, k] = dl_dalpha * (q[k] / t) * (ind - s_k)
            amb[i, k] = np.abs(p[k] - q[k]) <= NEAR_TIE * np.maximum(p[k], q[k])
    return grad, amb


# ---------------------------------------------------------------------------
# Small closed forms used by the speed model of the pages (context only)
# ---------------------------------------------------------------------------

def speedup_estimate(alpha, t_ar, t_draft, t_verify, t_overhead):
    """Single-user speedup: expected emitted tokens times the autoregressive
    step time, over the time of one draft/verify cycle.  The formula is lost
    on Speculative Decoding 与 MTP, section 7; this reading reproduces both of
    its printed examples."""
    return expected_emitted(alpha) * t_ar / (t_draft + t_verify + t_overhead)


# ---------------------------------------------------------------------------
# Verify-length scheduling over prefix survivals and a throughput table
# ---------------------------------------------------------------------------

# Relative gap below which two candidate throughputs count as a tie: another
# implementation's summation order may then pick the other one.
NEAR_SCHED = 1e-9


@dataclass
class ScheduleResult:
    lengths: np.ndarray  # int [R]: verify length l_r of every request
    theta: float         # tau * SPS(B) at the choice
    tau: float           # expected produced tokens
    batch: int           # B = sum_r (1 + l_r)
    near: bool           # another total length is within NEAR_SCHED of theta


def schedule_lengths(survival, sps):
    """Verify lengths that maximise the expected throughput.

    Bebop/DSpark blog, section "DSpark 的第二块拼图" and the equations after it:
    request r verifying l_r drafted tokens adds 1 + l_r tokens to the target
    batch, B = sum_r (1 + l_r); it produces tau_r = 1 + sum_{j<=l_r} a_{r,j}
    tokens in expectation, a_{r,j} the prefix survival; the throughput is
    Theta = (sum_r tau_r) * SPS(B), SPS(B) the decode steps per second at
    batch B (a measured table with steps and cliffs); the scheduler takes the
    argmax over l_1..l_R.

    survival: [R, L] a_{r,j} for j = 1..L (non-increasing in j as a product of
    per-position acceptances; the running minimum along j is used, which
    changes nothing for such input); sps: SPS(B) for B = 0, 1, ...,
    at least R * (1 + L).

    For a fixed B the best tau takes the B - R largest survivals (a row's
    survivals are non-increasing, so the chosen ones form a prefix of every
    row); the search is then over B.  Ties: equal survivals are taken in
    (row, position) order and equal throughputs keep the smaller B.
    """
    a = np.asarray(survival, dtype=np.float64)
    R, L = a.shape
    s = np.asarray(sps, dtype=np.float64)
    if s.shape[0] < R * (1 + L) + 1:
        raise ValueError("sps must cover B = 0 .. R * (1 + L)")
    a = np.minimum.accumulate(np.maximum(a, 0.0), axis=1)
    flat = a.reshape(-1)
    order = np.lexsort((np.arange(R * L), -flat))  # survival descending, then (row, position)
    vals = flat[order]
    best_m, best = 0, None
    thetas = []
    run = 0.0
    for m in range(R * L + 1):
        if m > 0:
            run += vals[m - 1]
        th = (R + run) * s[R + m]
        thetas.append(th)
        if best is None or th > best:
            best, best_m = th, m
    lengths = np.zeros(R, dtype=np.int64)
    for idx in order[:best_m]:
        lengths[idx // L] += 1
    tau = R + float(np.sum(vals[:best_m]))
    th = np.asarray(thetas)
    others = np.delete(th, best_m)
    near = bool(others.size and np.any(np.abs(others - best) <= NEAR_SCHED * max(abs(best), 1e-300)))
    return ScheduleResult(lengths, float(best), tau, int(R + best_m), near)
