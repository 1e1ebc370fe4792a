"""Plain, slow, float64 CPU oracle of the compression + decode path.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing on the product
path imports this module, and it shares no code with the CUDA library.

Sources (web pages, cited by title and section):

* [GK]  "GraceKV - Every Cache Entry Earns Its Place: Global Allocation of
        Resolution and Coverage for KV Cache Compression" (project page):
        sections "01 Curvature-guided partition", "02 Progressively refinable
        representation" / "Inside one cache entry", "03 Bottom-up value flow",
        "Exact-information safeguard", "04 Top-down budget flow",
        "05 Physical cache packing", "Technical details and default settings",
        and the budget-region strip under "Core idea".
* [DC]  "DistillCache: KL-Guided Adaptive KV-Cache Eviction for Memory-Efficient
        LLM Inference": section 3.1.1 (state space: the five token features),
        section 3.1.4 (the eviction error bound), Algorithm 1 (top-B pruning).

Where the pages leave a step open the oracle takes one stated reading; the
readings are numbered R1..R18 and listed in the repository's design notes.
Each function names the readings it uses.

Parity status: the scoring, hop, prototype, decode, pack and budget steps are
pinned by invariants and brute-force tests in ``tests/test_oracle_*.py``.  The
exact numeric values of the distortion/utility formula (R4) and of the hop
propagation (R2) are pinned only through their stated readings plus the
invariants listed there (no page prints a worked example of them).
"""
from __future__ import annotations

import heapq
import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

N_NODES = 15          # depth-3 binary midpoint tree: 1 + 2 + 4 + 8 prototype nodes (R3)
N_OPS = 16            # op 0 = Add(slot); op 1 + j = Split(node j)
FIRST_LEAF = 7        # nodes 7..14 are the leaf prototypes


# =============================================================================== RoPE
def rope_theta(d: int, base: float) -> np.ndarray:
    """theta_j = base^(-2j/d), j < d/2 (reading R9: rotate-half pairing)."""
    return base ** (-2.0 * np.arange(d // 2, dtype=np.float64) / d)


def rope_rotate(x: np.ndarray, pos, base: float) -> np.ndarray:
    """Rotate ``x[..., d]`` by RoPE at real-valued position(s) ``pos``.

    Pairing (j, j + d/2): out_j = x_j cos - x_{j+d/2} sin,
    out_{j+d/2} = x_{j+d/2} cos + x_j sin, angle = pos * theta_j.  A negative
    position is the inverse rotation.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None] * rope_theta(d, base)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# =============================================================================== a1: scoring
@dataclass
class HeadScores:
    lse: np.ndarray        # [R] log-sum-exp of each probe row
    H_rows: np.ndarray     # [R] entropy of each probe row's attention
    a: np.ndarray          # [R, n] attention probabilities
    feats: np.ndarray      # [n, 5] (alpha, |v|, sigma, H, pos)


def probe_attention(Kh: np.ndarray, Qh: np.ndarray, n: int, P: int) -> Tuple[np.ndarray, np.ndarray]:
    """Softmax attention of the probe rows over the keys, with the causal mask.

    [GK] "03 Bottom-up value flow": direct attention from the question /
    sequence-tail probes.  [DC] 3.1.1: the recent queries t-w+1..t.
    Rows are rho = g*P + p (query head g of this KV group, probe p).  Probe p
    sits at position n - P + p and sees keys i <= n - P + p (reading R15).
    Returns (scores s[R, n] with -inf where masked, lse[R]).
    """
    G = Qh.shape[0]
    d = Kh.shape[1]
    q = np.asarray(Qh, np.float64).reshape(G * P, d)
    s = q @ np.asarray(Kh, np.float64).T / math.sqrt(d)
    p_of_row = np.tile(np.arange(P), G)
    visible = np.arange(n)[None, :] <= (n - P + p_of_row)[:, None]
    s = np.where(visible, s, -np.inf)
    m = s.max(axis=1)
    lse = m + np.log(np.exp(s - m[:, None]).sum(axis=1))
    return s, lse


def score_head(Kh: np.ndarray, Vh: np.ndarray, Qh: np.ndarray, n: int, P: int) -> HeadScores:
    """Row statistics and the five per-token features of [DC] 3.1.1.

    alpha_i  = mean over probe rows of a_rho(i)
    |v_i|    = L2 norm of the value
    sigma_i  = population variance over the G query heads of mean_p a_{g,p}(i)
               (reading R14: "variance across heads" within the KV group)
    H_i      = sum_rho a_rho(i) H(a_rho) / sum_rho a_rho(i)
    pos_i    = i / (n - 1)
    """
    G = Qh.shape[0]
    s, lse = probe_attention(Kh, Qh, n, P)
    a = np.exp(s - lse[:, None])                       # masked entries -> exp(-inf) = 0
    with np.errstate(divide="ignore", invalid="ignore"):
        alog = np.where(a > 0, a * np.log(np.where(a > 0, a, 1.0)), 0.0)
    H_rows = -alog.sum(axis=1)
    alpha = a.mean(axis=0)
    vnorm = np.linalg.norm(np.asarray(Vh, np.float64), axis=1)
    mass = a.sum(axis=0)
    Hi = np.where(mass > 0, (a * H_rows[:, None]).sum(axis=0) / np.where(mass > 0, mass, 1.0), 0.0)
    mg = a.reshape(G, P, n).mean(axis=1)
    sigma = ((mg - mg.mean(axis=0)) ** 2).mean(axis=0)
    pos = np.arange(n, dtype=np.float64) / max(n - 1, 1)
    feats = np.stack([alpha, vnorm, sigma, Hi, pos], axis=1)
    return HeadScores(lse=lse, H_rows=H_rows, a=a, feats=feats)


# =============================================================================== a2: hops
def top_indices(x: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries, ties broken toward the lower index (R13)."""
    order = np.lexsort((np.arange(x.shape[0]), -x))
    return order[:k]


def hop_relevance(alpha: np.ndarray, Kh: np.ndarray, Vh: np.ndarray, S_h: int,
                  hop_weight: float, n_hops: int):
    """Two rounds of token-to-token relevance propagation ([GK] "03", defaults:
    two graph hops with weight 0.3), reading R2:

        r^0 = alpha
        seeds_k = the S_h tokens with the largest r^(k-1)
        Prop_j  = sum_{s in seeds_k} r^(k-1)_s * softmax_j(v_s . k_j / sqrt(d))   (all j < n)
        r^k     = r^0 + hop_weight * Prop

    Returns (r^(n_hops), list of seed index arrays).
    """
    K = np.asarray(Kh, np.float64)
    V = np.asarray(Vh, np.float64)
    d = K.shape[1]
    r0 = np.asarray(alpha, np.float64)
    r = r0.copy()
    seeds_all = []
    for _ in range(n_hops):
        seeds = top_indices(r, min(S_h, r.shape[0]))
        sc = V[seeds] @ K.T / math.sqrt(d)
        sc -= sc.max(axis=1, keepdims=True)
        A = np.exp(sc)
        A /= A.sum(axis=1, keepdims=True)
        prop = (r[seeds][:, None] * A).sum(axis=0)
        r = r0 + hop_weight * prop
        seeds_all.append(seeds)
    return r, seeds_all


# =============================================================================== a3: trees and prototypes
def tree_nodes(x: int, y: int, cuts: Optional[Sequence[int]] = None,
               extract: Optional[Sequence[int]] = None) -> List[Tuple[int, int]]:
    """The 15 prototype nodes of a slot [x, y) in breadth-first order (reading R3).

    Node j has children 2j+1 and 2j+2; a node [a, b) splits at floor((a+b)/2),
    or, when ``cuts`` is given, at the absolute position cuts[j] (j < 7; the
    curvature-chosen trees of reading R18).  Nodes 7..14 are the leaf
    prototypes; splitting one yields its tokens.  ``extract`` (reading R19)
    gives, per depth-2 node j = 3..6, the absolute position t of the salient
    token it isolates, or -1: such a node [a, b) has the three-way child set
    {[a, t), token t, [t+1, b)}, so its leaves are [a, t) and [t+1, b) and t
    belongs to no leaf.
    """
    nodes = [(x, y)]
    for j in range(7):
        a, b = nodes[j]
        t = -1 if extract is None or j < 3 else int(extract[j - 3])
        if t >= 0:
            if not extract_valid(t, a, b):
                raise ValueError(f"salient token {t} of node {j} invalid in [{a}, {b})")
            nodes.append((a, t))
            nodes.append((t + 1, b))
            continue
        mid = (a + b) // 2 if cuts is None else int(cuts[j])
        if not a < mid < b:
            raise ValueError(f"cut {mid} of node {j} outside ({a}, {b})")
        nodes.append((a, mid))
        nodes.append((mid, b))
    return nodes


SIDE_MIN = 2          # R19: each side span of a three-way child set keeps 2..15 tokens
SIDE_MAX = 15


def extract_valid(t: int, a: int, b: int) -> bool:
    """Whether token t may be isolated from node [a, b) (reading R19): both side
    spans [a, t) and [t+1, b) keep SIDE_MIN..SIDE_MAX tokens (a side of one
    token would be a prototype identical to its token, and a leaf holds at
    most 16 tokens)."""
    return SIDE_MIN <= t - a <= SIDE_MAX and SIDE_MIN <= b - t - 1 <= SIDE_MAX


def salient_tokens(r: np.ndarray, x0: int, y0: int, cuts: Optional[Sequence[int]] = None
                   ) -> List[int]:
    """The salient token each depth-2 node isolates (reading R19; [GK] "Technical
    details and default settings": tree construction may isolate a salient
    token with a three-way child set; "Exact-information safeguard": Split /
    Extract of a name-bearing span).  For depth-2 node j = 3..6 of the binary
    tree (midpoint or ``cuts``), t = the node's most relevant token (largest
    r_i, ties to the smaller i); the node isolates it when ``extract_valid``,
    else keeps its binary split (-1).  Comparisons only, in r's precision."""
    nodes = tree_nodes(x0, y0, cuts)
    out = []
    for j in range(3, 7):
        a, b = nodes[j]
        t = a + int(np.argmax(np.asarray(r[a:b])))
        out.append(t if extract_valid(t, a, b) else -1)
    return out


def node_parent(j: int) -> int:
    return -1 if j == 0 else (j - 1) // 2


@dataclass
class Prototype:
    k_hat: np.ndarray   # [d] post-RoPE key at the representative position
    v_hat: np.ndarray   # [d]
    log_m: float
    p_bar: float
    m: float
    kappa: float


def prototype(Kpost: np.ndarray, V: np.ndarray, r: np.ndarray, x: int, y: int,
              base: float, value_floor: float) -> Prototype:
    """One merged cache entry for tokens [x, y) ([GK] "Inside one cache entry").

    Key: inverse-rotate the post-RoPE keys to a shared frame, average, rotate
    again at the representative position p_bar = (x + y - 1) / 2 (R8).
    Multiplicity: m = c * clamp(kappa, 1/c, 1) with kappa the mean cosine of
    each unrotated key to the unrotated mean (R7).
    Value: weights w_i = (1 - f) r_i / sum r + f / c with f = value_floor
    (uniform weights when sum r = 0).
    """
    c = y - x
    pos = np.arange(x, y, dtype=np.float64)
    ktil = rope_rotate(Kpost, -pos, base)
    kbar = ktil.mean(axis=0)
    p_bar = (x + y - 1) / 2.0
    k_hat = rope_rotate(kbar, p_bar, base)
    nb = np.linalg.norm(kbar)
    nk = np.linalg.norm(ktil, axis=1)
    cos = np.where((nk > 0) & (nb > 0), (ktil @ kbar) / np.where(nk * nb > 0, nk * nb, 1.0), 0.0)
    kappa = float(cos.mean())
    m = c * min(max(kappa, 1.0 / c), 1.0)
    r = np.asarray(r, np.float64)
    rs = r.sum()
    w = (1.0 - value_floor) * r / rs + value_floor / c if rs > 0 else np.full(c, 1.0 / c)
    v_hat = w @ np.asarray(V, np.float64)
    return Prototype(k_hat=k_hat, v_hat=v_hat, log_m=math.log(m), p_bar=p_bar, m=m, kappa=kappa)


# =============================================================================== a4: distortion, value, utility
def node_distortion(a_node: np.ndarray, Vn: np.ndarray, q: np.ndarray, lse: np.ndarray,
                    proto: Prototype, nu_bar: float, w_part: float, w_value: float):
    """Probe-based fidelity of one prototype ([GK] technical details: attention-
    partition error and value-aggregate error weighed 0.25 : 0.75), reading R4.

    For each probe row rho:  A = sum_{i in N} a(i),  U = sum_{i in N} a(i) v_i,
    A_hat = exp(q . k_hat / sqrt(d) + log m - LSE),  U_hat = A_hat v_hat.
        D      = w_part mean|A - A_hat| + w_value mean|U - U_hat|_2 / nu_bar
        D_drop = w_part mean A          + w_value mean|U|_2 / nu_bar
    Returns (D, D_drop).
    """
    d = q.shape[1]
    A = a_node.sum(axis=1)
    U = a_node @ np.asarray(Vn, np.float64)
    A_hat = np.exp(q @ proto.k_hat / math.sqrt(d) + proto.log_m - lse)
    U_hat = A_hat[:, None] * proto.v_hat[None, :]
    part = np.abs(A - A_hat).mean()
    part_drop = A.mean()
    if nu_bar > 0:
        val = np.linalg.norm(U - U_hat, axis=1).mean() / nu_bar
        val_drop = np.linalg.norm(U, axis=1).mean() / nu_bar
    else:
        val = val_drop = 0.0
    return w_part * part + w_value * val, w_part * part_drop + w_value * val_drop


def gain_fraction(x: float, ddrop: float) -> float:
    """Fidelity gain as a fraction of the drop distortion, clamped to [0, 1] (R4)."""
    if not ddrop > 0:
        return 0.0
    return min(max(x / ddrop, 0.0), 1.0)


def slot_ops(D: np.ndarray, Ddrop: np.ndarray, Rv: np.ndarray, sizes: np.ndarray, sens: float,
             extract: Optional[Sequence[int]] = None):
    """Utilities and costs of the 16 ops of one slot tree ([GK] "04 Top-down
    budget flow": utility per entry = relevance x fidelity gain x head
    sensitivity / new physical entries).

    Add: cost 1, gain = 1 - D(root)/D_drop(root).
    Split(internal N): cost 1, gain = (D(N) - D(c1) - D(c2)) / D_drop(N).
    Split(depth-2 N with a three-way child set, reading R19): cost 2 (three
    entries replace one), gain = (D(N) - D(c1) - D(c2)) / D_drop(N) (the
    isolated token is exact, distortion 0).
    Split(leaf N of c tokens): cost c - 1, gain = D(N) / D_drop(N) (tokens are exact).
    Relevance of a node is the sum of its tokens' relevance ([GK] "03": parent
    value = sum of child values).
    """
    util = np.zeros(N_OPS, dtype=np.float64)
    cost = np.zeros(N_OPS, dtype=np.int64)
    cost[0] = 1
    util[0] = Rv[0] * gain_fraction(Ddrop[0] - D[0], Ddrop[0]) * sens
    for j in range(N_NODES):
        if j < FIRST_LEAF:
            c = 2 if (extract is not None and j >= 3 and extract[j - 3] >= 0) else 1
            g = gain_fraction(D[j] - D[2 * j + 1] - D[2 * j + 2], Ddrop[j])
        else:
            c = int(sizes[j]) - 1
            g = gain_fraction(D[j], Ddrop[j])
        cost[1 + j] = c
        util[1 + j] = Rv[j] * g * sens / c
    return util, cost


@dataclass
class HeadResult:
    lse: np.ndarray
    feats: np.ndarray
    r: np.ndarray
    seeds: List[np.ndarray]
    util: np.ndarray     # [S, 16] float64
    cost: np.ndarray     # [S, 16] int64
    D: np.ndarray        # [S, 15]
    Ddrop: np.ndarray    # [S, 15]
    protos: Optional[List[List[Prototype]]] = None
    Rv: Optional[np.ndarray] = None   # [S, 15] node values R(N), as used by the ops
    extract: Optional[np.ndarray] = None   # [S, 4] salient tokens (R19), -1 = none


def score_and_value_head(Kh, Vh, Qh, n: int, P: int, bounds: np.ndarray, sens: float,
                         base: float = 10000.0, hop_weight: float = 0.3, n_hops: int = 2,
                         w_part: float = 0.25, w_value: float = 0.75, value_floor: float = 0.1,
                         S_h: Optional[int] = None, keep_protos: bool = False,
                         cuts: Optional[np.ndarray] = None, salient: bool = False,
                         salient_r: Optional[np.ndarray] = None) -> HeadResult:
    """Everything the scoring call produces for one (layer, KV head): a1 -> a4.
    ``cuts`` [S, 7] gives the trees' cut positions (R18); None = midpoint trees.
    ``salient``: the depth-2 nodes isolate their salient tokens (R19), chosen on
    ``salient_r`` when given (e.g. the device's float32 relevance, for a
    bit-exact comparison of the choice), else on this oracle's relevance."""
    Kh = np.asarray(Kh, np.float64)
    Vh = np.asarray(Vh, np.float64)
    G = Qh.shape[0]
    d = Kh.shape[1]
    sc = score_head(Kh, Vh, Qh, n, P)
    S_h = P if S_h is None else S_h
    r, seeds = hop_relevance(sc.feats[:, 0], Kh, Vh, S_h, hop_weight, n_hops)
    q = np.asarray(Qh, np.float64).reshape(G * P, d)
    nu_bar = float(sc.feats[:, 1].mean())
    S = len(bounds) - 1
    util = np.zeros((S, N_OPS))
    cost = np.zeros((S, N_OPS), dtype=np.int64)
    Dall = np.zeros((S, N_NODES))
    Rall = np.zeros((S, N_NODES))
    Ddall = np.zeros((S, N_NODES))
    ext_all = np.full((S, 4), -1, dtype=np.int64)
    protos_all = []
    for s in range(S):
        x0, y0 = int(bounds[s]), int(bounds[s + 1])
        cs = None if cuts is None else cuts[s]
        ext = None
        if salient:
            ext = salient_tokens(r if salient_r is None else salient_r, x0, y0, cs)
            ext_all[s] = ext
        nodes = tree_nodes(x0, y0, cs, ext)
        D = np.zeros(N_NODES)
        Dd = np.zeros(N_NODES)
        Rv = np.zeros(N_NODES)
        sizes = np.zeros(N_NODES, dtype=np.int64)
        plist = []
        for j, (x, y) in enumerate(nodes):
            pr = prototype(Kh[x:y], Vh[x:y], r[x:y], x, y, base, value_floor)
            D[j], Dd[j] = node_distortion(sc.a[:, x:y], Vh[x:y], q, sc.lse, pr, nu_bar,
                                          w_part, w_value)
            Rv[j] = r[x:y].sum()
            sizes[j] = y - x
            plist.append(pr)
        util[s], cost[s] = slot_ops(D, Dd, Rv, sizes, sens, ext)
        Dall[s], Ddall[s], Rall[s] = D, Dd, Rv
        if keep_protos:
            protos_all.append(plist)
    return HeadResult(lse=sc.lse, feats=sc.feats, r=r, seeds=seeds, util=util, cost=cost,
                      D=Dall, Ddrop=Ddall, protos=protos_all if keep_protos else None, Rv=Rall,
                      extract=ext_all if salient else None)


# =============================================================================== f3: curvature-chosen trees
LEAF_MIN = 2          # R18: a cut keeps every leaf prototype at 2..16 tokens, the range of
LEAF_MAX = 16         # the midpoint trees' leaves over slots of 16..128 tokens


def key_curvature(Kh: np.ndarray, base: float, scales: Sequence[int] = (1, 2, 4, 8)) -> np.ndarray:
    """Curvature of one (layer, KV head)'s key trajectory (reading R18).

    [GK] "01 Curvature-guided partition" measures where a normalized trajectory
    turns; the tree of a (layer, KV head, slot) is cut with the same measure
    taken on that head's own keys with RoPE removed (k~_i = R(-i) k_i, so the
    position rotation itself is no turn): the multi-scale curvature of
    ``curvature`` on the rows k~_i."""
    Kh = np.asarray(Kh, np.float64)
    u = rope_rotate(Kh, -np.arange(Kh.shape[0], dtype=np.float64), base)
    return curvature(u, scales)


def tree_cuts(kappa: np.ndarray, x0: int, y0: int, dtype=np.float64) -> List[int]:
    """Cut positions of the 7 internal nodes (breadth-first) of slot [x0, y0)
    ([GK] "Technical details": tree construction considers high-curvature split
    candidates plus the midpoint), reading R18.

    Top-down, node [a, b) of depth k (c = b - a tokens, midpoint m =
    floor((a+b)/2)) is cut at the valid t maximising
        score(t) = kappa[t] - lam * ((t - m) / (c / 2))^2,   lam = mean kappa[a:b)
    (the partition's curvature gain with its length-balance penalty, so the
    midpoint, penalty 0, wins unless a turn outweighs its imbalance).  A cut at
    t makes children [a, t) and [t, b); it is valid when each child keeps
    LEAF_MIN..LEAF_MAX tokens per leaf below it (2^(2-k) leaves), so a leaf
    split always stores at least 2 tokens for its cost; the midpoint of every
    node of a slot of 16..128 tokens always is valid.  Ties go to the midpoint,
    then to the smaller t.  Every operation is
    rounded to ``dtype`` in the order written (lam summed in index order), so
    ``dtype=np.float32`` reproduces a single-precision evaluation exactly.
    """
    f = np.dtype(dtype).type
    k = np.asarray(kappa).astype(dtype)
    nodes = [(x0, y0)]
    cuts = []
    for j in range(7):
        a, b = nodes[j]
        depth = 0 if j == 0 else (1 if j < 3 else 2)
        lo = LEAF_MIN * 2 ** (2 - depth)
        hi = LEAF_MAX * 2 ** (2 - depth)
        c = b - a
        m = (a + b) // 2
        acc = f(0)
        for i in range(a, b):
            acc = f(acc + k[i])
        lam = f(acc / f(c))
        half = f(f(c) * f(0.5))

        def score(t):
            r = f(f(t - m) / half)
            return f(k[t] - f(lam * f(r * r)))

        best_t, best = m, score(m)
        for t in range(a + lo, b - lo + 1):
            if not (lo <= t - a <= hi and lo <= b - t <= hi):
                continue
            sc = score(t)
            if sc > best:
                best_t, best = t, sc
        cuts.append(best_t)
        nodes.append((a, best_t))
        nodes.append((best_t, b))
    return cuts


def slot_cuts(kappa: np.ndarray, bounds: np.ndarray, dtype=np.float64) -> np.ndarray:
    """``tree_cuts`` of every slot of one (layer, KV head): [S, 7] absolute positions."""
    S = len(bounds) - 1
    return np.asarray([tree_cuts(kappa, int(bounds[s]), int(bounds[s + 1]), dtype)
                       for s in range(S)], dtype=np.int64).reshape(S, 7)


# =============================================================================== a5: budget, floor, auction
def budget(n: int, L: int, H: int, W: int, budget_ratio: float, budget_entries_per_lh: int,
           floor_cap_frac: float):
    """Physical budget of one sequence ([GK] "Core idea": one stored K/V pair is
    one budget unit; the recent window is exact and counts toward the budget).

    B_tot = floor(beta * n) * L * H (or entries_per_lh * L * H), reading R11;
    B_alloc = B_tot - W * L * H; floor cap = floor(frac * B_alloc) entries (R6).
    """
    per_lh = budget_entries_per_lh if budget_entries_per_lh > 0 else int(math.floor(budget_ratio * n))
    B_tot = per_lh * L * H
    B_alloc = B_tot - W * L * H
    if B_alloc < 0:
        raise ValueError("budget smaller than the recent window")
    cap = int(math.floor(floor_cap_frac * B_alloc))
    return B_tot, B_alloc, cap


def _leaf_of(i: int, x0: int, y0: int, cuts=None, extract=None) -> Tuple[int, List[int]]:
    """The node whose split makes token i exact (its leaf, or the depth-2 node
    that isolates it, reading R19) and the node path root..that node."""
    nodes = tree_nodes(x0, y0, cuts, extract)
    j = 0
    path = [0]
    while j < FIRST_LEAF:
        if extract is not None and j >= 3 and int(extract[j - 3]) == i:
            return j, path
        c1 = 2 * j + 1
        j = c1 if i < nodes[c1][1] else c1 + 1
        path.append(j)
    return j, path


@dataclass
class Selection:
    taken: np.ndarray        # bool [L, H, S, 16]
    floor_spent: int
    floor_tokens: int
    auction_spent: int
    B_tot: int
    B_alloc: int
    lens: np.ndarray         # int [L, H] entries per (l, h) incl. window


def singleton_floor(r: np.ndarray, sens: np.ndarray, bounds: np.ndarray, cost: np.ndarray,
                    cap_entries: int, cap_tokens: int, taken: np.ndarray,
                    cuts: Optional[np.ndarray] = None, extract: Optional[np.ndarray] = None):
    """Capped singleton floor before the auction ([GK] "Exact-information
    safeguard" and technical details), reading R6.

    Candidates: every compressible (l, h, i) with r_i > 0, in order of
    (r_i * sens[l, h] descending, (l, h, i) ascending).  A candidate's path is
    Add(slot), Split of each ancestor, Split of its leaf prototype; its cost is
    the cost of the path ops not yet taken (shared ancestors paid once).  A
    token already exact is skipped at no cost.  If the path fits in the cap it
    is taken and the token counted, otherwise the floor stops; it also stops
    once cap_tokens tokens are counted (cap_tokens < 0: no token cap).
    The key r * sens is computed in the precision of ``r``.  ``cuts`` [L, H,
    S, 7] gives the trees' cut positions (R18); None = midpoint trees.
    ``extract`` [L, H, S, 4]: the salient tokens the depth-2 nodes isolate
    (R19; -1 = none): such a token's path ends at its depth-2 node's split.
    Mutates ``taken`` and returns (spent, tokens).
    """
    L, H, n_ = r.shape
    end = int(bounds[-1])
    S = len(bounds) - 1
    keys = r[:, :, :end] * sens.astype(r.dtype)[:, :, None]
    keys = keys.astype(r.dtype)
    flat = keys.reshape(-1)
    lhs = np.repeat(np.arange(L * H), end)
    ii = np.tile(np.arange(end), L * H)
    cand = (r[:, :, :end].reshape(-1) > 0)
    cidx = lhs.astype(np.int64) * n_ + ii
    sel = np.nonzero(cand)[0]
    order = sel[np.lexsort((cidx[sel], -flat[sel].astype(np.float64)))]
    slot_of = np.searchsorted(bounds, np.arange(end), side="right") - 1
    spent = 0
    tokens = 0
    for k in order:
        if cap_tokens >= 0 and tokens >= cap_tokens:
            break
        lh = int(lhs[k]); i = int(ii[k])
        l, h = divmod(lh, H)
        s = int(slot_of[i])
        x0, y0 = int(bounds[s]), int(bounds[s + 1])
        leaf, path = _leaf_of(i, x0, y0, None if cuts is None else cuts[l, h, s],
                              None if extract is None else extract[l, h, s])
        t = taken[l, h, s]
        if t[1 + leaf]:
            continue                                   # already exact
        ops = [0] + [1 + j for j in path]
        c = sum(int(cost[l, h, s, o]) for o in ops if not t[o])
        if spent + c <= cap_entries:
            for o in ops:
                t[o] = True
            spent += c
            tokens += 1
        else:
            break
    return spent, tokens


def op_parent(o: int) -> int:
    """Op whose taking exposes op o (-1 for Add)."""
    if o == 0:
        return -1
    j = o - 1
    return 0 if j == 0 else 1 + node_parent(j)


def greedy_auction(util: np.ndarray, cost: np.ndarray, taken: np.ndarray, remaining: int) -> int:
    """Global greedy Add/Split auction ([GK] "04 Top-down budget flow").

    One queue holds every exposed op of every (l, h, slot): Add for an absent
    slot, Split for a present, unsplit prototype.  Repeatedly pop the highest
    (utility desc, op id asc) op; if its cost fits in the remaining budget take
    it and expose its children's Splits, otherwise discard it (its subtree is
    never exposed).  Runs until the queue is empty; zero-utility ops are still
    bought while budget lasts.  Op id = ((l*H + h)*S + slot)*16 + local.
    Mutates ``taken``; returns the entries spent.
    """
    L, H, S, _ = util.shape
    heap = []

    def push(l, h, s, o):
        gid = ((l * H + h) * S + s) * N_OPS + o
        heapq.heappush(heap, (-float(util[l, h, s, o]), gid, l, h, s, o))

    for l in range(L):
        for h in range(H):
            for s in range(S):
                t = taken[l, h, s]
                if not t[0]:
                    push(l, h, s, 0)
                    continue
                for j in range(N_NODES):
                    present = t[0] if j == 0 else t[1 + node_parent(j)]
                    if present and not t[1 + j]:
                        push(l, h, s, 1 + j)
    spent = 0
    while heap:
        _, _, l, h, s, o = heapq.heappop(heap)
        c = int(cost[l, h, s, o])
        if c <= remaining:
            taken[l, h, s, o] = True
            remaining -= c
            spent += c
            if o == 0:
                push(l, h, s, 1)
            else:
                j = o - 1
                if j < FIRST_LEAF:
                    push(l, h, s, 1 + 2 * j + 1)
                    push(l, h, s, 1 + 2 * j + 2)
    return spent


def full_heads(r: np.ndarray, end: int, frac: float) -> np.ndarray:
    """Head-level hybrid ([DC] App. E.3: the top 20% of heads by an attention
    statistic keep the full cache), reading R16: the statistic of (l, h) is its
    relevance mass outside the recent window, sum of r_i over i < end, summed in
    float64 over the float32 relevances; the floor(frac * L * H) heads with the
    largest statistic (ties: lower l*H + h first) are full.  Returns bool [L, H]."""
    L, H, _ = r.shape
    F = int(math.floor(frac * L * H))
    imp = np.asarray(r[:, :, :end], dtype=np.float64).sum(axis=-1).reshape(-1)
    order = np.lexsort((np.arange(L * H), -imp))
    full = np.zeros(L * H, dtype=bool)
    full[order[:F]] = True
    return full.reshape(L, H)


def select_sequence(util: np.ndarray, cost: np.ndarray, r: np.ndarray, sens: np.ndarray,
                    bounds: np.ndarray, n: int, W: int, budget_ratio: float,
                    budget_entries_per_lh: int, floor_cap_frac: float, floor_cap_tokens: int,
                    head_full_frac: float = 0.0, cuts: Optional[np.ndarray] = None,
                    extract: Optional[np.ndarray] = None) -> Selection:
    """Budget -> singleton floor -> greedy auction for one sequence (a5).

    With head_full_frac > 0 (the head-level hybrid, R16) the full heads store
    every token exact (all ops taken, len = n) and pay n - W beyond their
    window from the same budget; the floor and the auction run on the other
    heads with B_alloc = B_tot - W*L*H - F*(n - W) and the floor cap taken of
    that reduced pool.  ``cuts`` [L, H, S, 7]: the trees' cut positions (R18);
    ``extract`` [L, H, S, 4]: the depth-2 nodes' isolated salient tokens (R19)."""
    L, H, S, _ = util.shape
    B_tot, B_alloc, cap = budget(n, L, H, W, budget_ratio, budget_entries_per_lh, floor_cap_frac)
    taken = np.zeros((L, H, S, N_OPS), dtype=bool)
    if head_full_frac > 0:
        full = full_heads(r, int(bounds[-1]), head_full_frac)
        taken[full] = True
        B_alloc -= int(full.sum()) * (n - W)
        if B_alloc < 0:
            raise ValueError("budget smaller than the full heads and the windows")
        cap = int(math.floor(floor_cap_frac * B_alloc))
    fs, ft = singleton_floor(r, sens, bounds, cost, min(cap, B_alloc), floor_cap_tokens, taken,
                             cuts, extract)
    asp = greedy_auction(util, cost, taken, B_alloc - fs)
    lens = W + (taken * cost).sum(axis=(2, 3))
    return Selection(taken=taken, floor_spent=fs, floor_tokens=ft, auction_spent=asp,
                     B_tot=B_tot, B_alloc=B_alloc, lens=lens.astype(np.int64))


# =============================================================================== a6: pack
def frontier(t: np.ndarray, x0: int, y0: int, cuts=None, extract=None) -> List[Tuple[str, int]]:
    """Stored entries of one slot tree, left to right ([GK] "05 Physical cache
    packing"): an absent root stores nothing, a present unsplit node stores its
    prototype, a split leaf prototype stores its tokens exactly, and a split
    depth-2 node with a three-way child set (R19) stores its left side, its
    salient token exactly, then its right side."""
    nodes = tree_nodes(x0, y0, cuts, extract)

    def visit(j):
        if not t[1 + j]:
            return [("node", j)]
        if extract is not None and 3 <= j < FIRST_LEAF and extract[j - 3] >= 0:
            return visit(2 * j + 1) + [("tok", int(extract[j - 3]))] + visit(2 * j + 2)
        if j < FIRST_LEAF:
            return visit(2 * j + 1) + visit(2 * j + 2)
        a, b = nodes[j]
        return [("tok", i) for i in range(a, b)]

    return visit(0) if t[0] else []


@dataclass
class Packed:
    K: List[np.ndarray]      # per (b, l, h) flattened index: [len, d]
    V: List[np.ndarray]
    logm: List[np.ndarray]
    pos: List[np.ndarray]
    lens: np.ndarray         # [B, L, H]
    caps: np.ndarray         # [B, L, H]
    offs: np.ndarray         # [B, L, H] exclusive prefix sum of caps in (b, l, h) order


def pack_head(Kh, Vh, r, bounds, t_lh, n: int, W: int, base: float, value_floor: float,
              cuts: Optional[np.ndarray] = None, extract: Optional[np.ndarray] = None):
    """Entries of one (l, h): slots ascending, frontier left to right, then the
    window tokens [n - W, n).  Exact tokens keep their K/V and get log m = 0.
    ``cuts`` [S, 7] (R18), ``extract`` [S, 4] (R19) describe the trees."""
    Kh = np.asarray(Kh, np.float64)
    Vh = np.asarray(Vh, np.float64)
    ks, vs, lm, ps = [], [], [], []
    for s in range(len(bounds) - 1):
        x0, y0 = int(bounds[s]), int(bounds[s + 1])
        cs = None if cuts is None else cuts[s]
        es = None if extract is None else extract[s]
        nodes = tree_nodes(x0, y0, cs, es)
        for kind, j in frontier(t_lh[s], x0, y0, cs, es):
            if kind == "tok":
                ks.append(Kh[j]); vs.append(Vh[j]); lm.append(0.0); ps.append(float(j))
            else:
                x, y = nodes[j]
                pr = prototype(Kh[x:y], Vh[x:y], r[x:y], x, y, base, value_floor)
                ks.append(pr.k_hat); vs.append(pr.v_hat); lm.append(pr.log_m); ps.append(pr.p_bar)
    for i in range(n - W, n):
        ks.append(Kh[i]); vs.append(Vh[i]); lm.append(0.0); ps.append(float(i))
    d = Kh.shape[1]
    return (np.asarray(ks).reshape(-1, d), np.asarray(vs).reshape(-1, d),
            np.asarray(lm, np.float64), np.asarray(ps, np.float64))


def offsets(lens: np.ndarray, reserve: int):
    caps = lens + reserve
    flat = caps.reshape(-1)
    offs = np.concatenate([[0], np.cumsum(flat)[:-1]]).reshape(caps.shape)
    return caps, offs


# =============================================================================== a7: decode
def decode_head(q: np.ndarray, Kp: np.ndarray, Vp: np.ndarray, logm: np.ndarray) -> np.ndarray:
    """GQA attention of the G query heads of one KV head over its ragged entries
    with the +log m multiplicity bias ([GK] "Inside one cache entry", "05")."""
    q = np.asarray(q, np.float64)
    d = q.shape[-1]
    s = q @ np.asarray(Kp, np.float64).T / math.sqrt(d) + np.asarray(logm, np.float64)[None, :]
    s -= s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return p @ np.asarray(Vp, np.float64)


def decode_step_head(q, k_new, v_new, Kp, Vp, logm):
    """Append (k_new, v_new) with multiplicity 1, then attend over all entries
    including it (reading R10).  Returns (out [G, d], Kp', Vp', logm')."""
    Kp2 = np.concatenate([np.asarray(Kp, np.float64), np.asarray(k_new, np.float64)[None]], 0)
    Vp2 = np.concatenate([np.asarray(Vp, np.float64), np.asarray(v_new, np.float64)[None]], 0)
    lm2 = np.concatenate([np.asarray(logm, np.float64), [0.0]])
    return decode_head(q, Kp2, Vp2, lm2), Kp2, Vp2, lm2


# =============================================================================== f2: per-step top-B eviction
def evict_budget(n_seen: int, ratio: float, b_min: int) -> int:
    """[DC] Algorithm 1: B = max(floor(r * |C_t|), B_min); reading R17: |C_t| is the
    unpruned cache size, i.e. the tokens seen so far (prompt and generated,
    including this step's)."""
    return max(int(math.floor(ratio * n_seen)), b_min)


def evict_step(q: np.ndarray, k_new: np.ndarray, v_new: np.ndarray, K: np.ndarray, V: np.ndarray,
               n_seen: int, ratio: float, b_min: int):
    """One DistillCache inference step with the heuristic score s_i = alpha_i ([DC]
    Algorithm 1 and 3.1.1; the learned policy is replaced by its first feature,
    reading R17).  One sequence: K, V [L, H, c, d] hold the same c tokens in every
    (layer, KV head); q [L, H*G, d]; k_new, v_new [L, H, d].

    The new token is appended to every (l, h); every query head attends over
    the c + 1 entries (fp64 softmax); alpha_i = mean over (l, h, g) of the
    attention probability of entry i; B = evict_budget(n_seen, ...); the kept
    entries are the top-B by alpha (ties: lower cache index), in cache order.
    Returns (out [L, H*G, d], alpha [c + 1], keep [min(B, c + 1)] cache indices).
    """
    L, H, c, d = K.shape
    G = q.shape[1] // H
    q = np.asarray(q, np.float64)
    out = np.zeros((L, H * G, d))
    alpha = np.zeros(c + 1)
    for l in range(L):
        for h in range(H):
            Kc = np.concatenate([np.asarray(K[l, h], np.float64), np.asarray(k_new[l, h], np.float64)[None]])
            Vc = np.concatenate([np.asarray(V[l, h], np.float64), np.asarray(v_new[l, h], np.float64)[None]])
            sc = q[l, h * G:(h + 1) * G] @ Kc.T / math.sqrt(d)
            sc -= sc.max(axis=1, keepdims=True)
            pr = np.exp(sc)
            pr /= pr.sum(axis=1, keepdims=True)
            out[l, h * G:(h + 1) * G] = pr @ Vc
            alpha += pr.sum(axis=0)
    alpha /= L * H * G
    B = evict_budget(n_seen, ratio, b_min)
    keep = top_b(alpha, B)
    return out, alpha, keep


def top_b(score: np.ndarray, B: int) -> np.ndarray:
    """Indices of the B largest scores (ties: lower index first), ascending."""
    order = np.lexsort((np.arange(len(score)), -np.asarray(score, np.float64)))
    return np.sort(order[:min(B, len(score))])


# =============================================================================== a0: partition
def curvature(hidden: np.ndarray, scales: Sequence[int] = (1, 2, 4, 8)) -> np.ndarray:
    """Multi-scale curvature of the normalized hidden-state trajectory ([GK]
    "01 Curvature-guided partition"), reading R1:
    kappa_w(t) = 1 - cos(h_t - h_{t-w}, h_{t+w} - h_t), averaged over the
    scales w that fit (0 where none fits)."""
    h = np.asarray(hidden, np.float64)
    h = h / np.linalg.norm(h, axis=1, keepdims=True)
    n = h.shape[0]
    tot = np.zeros(n)
    cnt = np.zeros(n)
    for w in scales:
        if n <= 2 * w:
            continue
        a = h[w:n - w] - h[:n - 2 * w]
        b = h[2 * w:] - h[w:n - w]
        na = np.linalg.norm(a, axis=1)
        nb = np.linalg.norm(b, axis=1)
        cos = np.where(na * nb > 0, (a * b).sum(1) / np.where(na * nb > 0, na * nb, 1.0), 1.0)
        tot[w:n - w] += 1.0 - cos
        cnt[w:n - w] += 1
    return np.where(cnt > 0, tot / np.maximum(cnt, 1), 0.0)


def partition_dp(kappa: np.ndarray, end: int, lmin: int = 16, lmax: int = 128,
                 target: int = 64, lam: Optional[float] = None) -> np.ndarray:
    """Dynamic program over cut positions in [0, end) (reading R1).

    Maximise sum over interior cuts c of kappa(c) - lam * sum over slots of
    ((len - target) / target)^2, with lmin <= len <= lmax; lam defaults to the
    mean of kappa over [0, end).  Ties go to the smaller previous cut.
    """
    k = np.asarray(kappa, np.float64)
    if lam is None:
        lam = float(k[:end].mean()) if end > 0 else 0.0
    NEG = -np.inf
    best = np.full(end + 1, NEG)
    prev = np.full(end + 1, -1, dtype=np.int64)
    best[0] = 0.0
    for y in range(1, end + 1):
        gain_cut = k[y] if y < end else 0.0
        for ln in range(lmin, lmax + 1):
            x = y - ln
            if x < 0:
                break
            if best[x] == NEG:
                continue
            v = best[x] - lam * ((ln - target) / target) ** 2 + gain_cut
            if v > best[y] or (v == best[y] and x < prev[y]):
                best[y] = v
                prev[y] = x
    if best[end] == NEG:
        raise ValueError("no feasible partition")
    cuts = [end]
    y = end
    while y > 0:
        y = int(prev[y])
        cuts.append(y)
    return np.asarray(cuts[::-1], dtype=np.int32)
