"""Seeded synthetic inputs for the verify step.

This module is shared by the tests and the benchmark.  It holds no verify arithmetic (no
normalisation, acceptance test, residual or tree walk): it draws logits, uniforms, draft tokens and
tree shapes from fixed seeds.  Draft tokens stand in for the draft model's own sampler (the
proposal side, which sits outside the verify step): they are drawn by the Gumbel-max trick from the
stored draft logits, restricted to the draft's top-k set when top-k is on, so each token is a draw
from exactly the processed q that the verify step is told sampled it.

Workload recipes (five named configurations):

  c1  B=1   gamma=4 V=32     fp32  T=1.0  target N(0,2^2); draft = target + N(0,0.5^2)
  c2  B=8   gamma=4 V=32000  bf16  T=1.0  target N(0,3^2), 20 random peak tokens per row +8;
                                          draft = target + N(0,1^2)
  c3  B=64  gamma=5 V=128256 bf16  T=0.7  target N(0,3^2) + Zipf(1.1) rank bias -1.1*ln(rank);
                                          draft = 0.8*target + N(0,1.5^2)
  c4  B=256 gamma=7 V=152064 bf16  T=0.8  as c2 with draft noise N(0,2^2); top_k=50
  c5  B=32  N=64    V=128256 bf16         tree logits as c3's target, Medusa tree 4/4/2/2 in BFS
                                          order truncated to 64 nodes; a node's token is its
                                          predictor row's argmax with prob 0.6, else uniform
  c6  B=32  N=64    V=128256 bf16  T=0.7  stochastic tree verify: c5's tree; target rows as c3's
                                          target, draft rows = 0.8*target + N(0,1.5^2) laid out
                                          like the target rows (row 0 frontier, row i+1 at node i);
                                          the children of a node are i.i.d. draws from the draft
                                          row at their parent (qrow = parent + 1)
  c8  B=64  gamma=5 V=128256 bf16         linear greedy verify: c5's recipe on a chain of 5 drafted
                                          tokens (target rows as c3's target; a token is its row's
                                          argmax with prob 0.6, else uniform)
  c9  B=64  gamma=5 V=128256 bf16  T=0.7  grammar-masked verify: c3's logits; every position has its
                                          own valid-token set, one of three kinds with equal odds:
                                          narrow (64 random tokens), half (each token with
                                          probability 1/2), wide (each token blocked with
                                          probability 1/100); draft tokens from the masked q
  c10 B=32  N=64    V=128256 bf16  T=0.7  typical-acceptance tree verify: c5's recipe (tree, logits,
                                          tokens); eps = 0.09, delta = 0.3; one uniform per
                                          request for the token after the path
  c11 B=64  gamma=5 V=128256 bf16 T=0.8  top-p verify, top_p = 0.9 on every row: c2's target recipe
                                          (20 peak tokens per row +8) at c3's sizes, draft noise
                                          N(0,1^2); draft tokens from the draft's own nucleus
  c7  G=8 x N=8 particles, K=5, V=128256 bf16, T=0.7, eta = N/2: one SMC-SD round; logits as
                                          c3 (target, draft = 0.8*target + N(0,1.5^2)), draft
                                          tokens from q, incoming log weights N(0, 0.5^2),
                                          uniforms [B, 2] (extension, ancestor)

Streams: SeedSequence(seed).spawn(3) gives (logits, draft sampling, uniforms); each is spawned again
per request, so a request's inputs do not depend on B or on how many threads generate them.
Logits are drawn in float64, rounded to float32, and (for bf16) rounded to nearest-even bf16 bits;
the draft is built from the float32 target before rounding.  Uniforms are (uint32 >> 8) * 2^-24,
exact in float32 and in [0, 1).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np


# ------------------------------------------------------------------ configurations

@dataclass(frozen=True)
class SpecConfig:
    name: str
    B: int
    gamma: int
    V: int
    dtype: str          # "bf16" or "f32"
    temperature: float
    top_k: int          # 0 = off
    target: str         # "normal2" | "peaks" | "zipf"
    draft_scale: float  # draft = draft_scale * target + N(0, draft_noise^2)
    draft_noise: float
    seed: int
    mask: str = ""      # "" = no grammar mask; "grammar" = the mixed valid-set recipe (c9)
    top_p: float = 1.0  # < 1: the top-p processor on every row (c11)


@dataclass(frozen=True)
class TreeConfig:
    name: str
    B: int
    V: int
    branching: tuple = (4, 4, 2, 2)
    max_nodes: int = 64
    dtype: str = "bf16"
    p_match: float = 0.6
    seed: int = 1005
    chain: bool = False    # verified as a linear draft (spec_verify_greedy), not as a tree
    typical: bool = False  # verified by typical acceptance (tree_verify_typical)
    temperature: float = 0.7
    eps: float = 0.09      # typical acceptance: p(x) > min(eps, delta exp(-H))
    delta: float = 0.3


CONFIGS = {
    "c1": SpecConfig("c1", 1, 4, 32, "f32", 1.0, 0, "normal2", 1.0, 0.5, 1001),
    "c2": SpecConfig("c2", 8, 4, 32000, "bf16", 1.0, 0, "peaks", 1.0, 1.0, 1002),
    "c3": SpecConfig("c3", 64, 5, 128256, "bf16", 0.7, 0, "zipf", 0.8, 1.5, 1003),
    "c4": SpecConfig("c4", 256, 7, 152064, "bf16", 0.8, 50, "peaks", 1.0, 2.0, 1004),
}
TOPP_CONFIGS = {
    "c11": SpecConfig("c11", 64, 5, 128256, "bf16", 0.8, 0, "peaks", 1.0, 1.0, 1011, top_p=0.9),
}
MASK_CONFIGS = {
    "c9": SpecConfig("c9", 64, 5, 128256, "bf16", 0.7, 0, "zipf", 0.8, 1.5, 1009, mask="grammar"),
}
TREE_CONFIGS = {"c5": TreeConfig("c5", 32, 128256),
                "c8": TreeConfig("c8", 64, 128256, branching=(1, 1, 1, 1, 1), max_nodes=5,
                                 seed=1008, chain=True),
                "c10": TreeConfig("c10", 32, 128256, seed=1010, typical=True)}


@dataclass(frozen=True)
class SampleTreeConfig:
    name: str
    B: int
    V: int
    branching: tuple = (4, 4, 2, 2)
    max_nodes: int = 64
    dtype: str = "bf16"
    temperature: float = 0.7
    draft_scale: float = 0.8
    draft_noise: float = 1.5
    seed: int = 1006


SAMPLE_TREE_CONFIGS = {"c6": SampleTreeConfig("c6", 32, 128256)}


@dataclass(frozen=True)
class SmcConfig:
    name: str
    groups: int
    particles: int
    K: int
    V: int
    dtype: str = "bf16"
    temperature: float = 0.7
    eta: float = 4.0
    draft_scale: float = 0.8
    draft_noise: float = 1.5
    logw_sd: float = 0.5
    seed: int = 1007

    @property
    def B(self) -> int:
        return self.groups * self.particles


SMC_CONFIGS = {"c7": SmcConfig("c7", 8, 8, 5, 128256)}


def scaled(cfg, **kw):
    """A copy of a configuration with some fields replaced (smaller B, ragged V, ...)."""
    d = dict(cfg.__dict__)
    d.update(kw)
    return type(cfg)(**d)


# ------------------------------------------------------------------ primitives

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def stored_to_f64(a: np.ndarray) -> np.ndarray:
    """Stored logits (float32, or bf16 bits in uint16) as float64 values."""
    if a.dtype == np.uint16:
        return bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


def uniforms_from(rng: np.random.Generator, shape) -> np.ndarray:
    """(uint32 >> 8) * 2^-24: 24-bit uniforms, exact in float32, in [0, 1)."""
    w = rng.integers(0, 2**32, size=shape, dtype=np.uint64).astype(np.uint32)
    return ((w >> np.uint32(8)).astype(np.float64) * 2.0**-24).astype(np.float32)


def _store(x32: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x32) if dtype == "bf16" else np.ascontiguousarray(x32, np.float32)


def _zipf_bias(V: int, seed: int) -> np.ndarray:
    """bias_v = -1.1 * ln(rank_v) with rank a seeded global permutation of 1..V."""
    rank = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7]))).permutation(V) + 1
    return -1.1 * np.log(rank.astype(np.float64))


def _target_rows(rng: np.random.Generator, kind: str, rows: int, V: int, bias) -> np.ndarray:
    if kind == "normal2":
        t = rng.standard_normal((rows, V)) * 2.0
    elif kind == "peaks":
        t = rng.standard_normal((rows, V)) * 3.0
        for r in range(rows):
            t[r, rng.choice(V, size=min(20, V), replace=False)] += 8.0
    elif kind == "zipf":
        t = rng.standard_normal((rows, V)) * 3.0 + bias[None, :]
    else:
        raise ValueError(kind)
    return t.astype(np.float32)


def gumbel_max_tokens(rng: np.random.Generator, z: np.ndarray, keep: np.ndarray | None = None):
    """One categorical draw per row of softmax(z) (restricted to ``keep``) by the Gumbel-max trick."""
    g = z + rng.gumbel(size=z.shape)
    if keep is not None:
        g = np.where(keep, g, -np.inf)
    return np.argmax(g, axis=-1).astype(np.int32)


def draft_keep_mask(x: np.ndarray, top_k: int) -> np.ndarray | None:
    """The draft sampler's own top-k set: stored logit >= its k-th largest (ties kept)."""
    V = x.shape[-1]
    if not (0 < top_k < V):
        return None
    kth = -np.partition(-x, top_k - 1, axis=-1)[..., top_k - 1:top_k]
    return x >= kth


def grammar_valid_sets(rng: np.random.Generator, positions: int, V: int) -> np.ndarray:
    """Valid-token sets of ``positions`` grammar states, bool [positions, V].

    Each state is one of three kinds with equal odds: narrow (64 distinct random tokens, or all of
    them when V <= 64), half (each token valid with probability 1/2) or wide (each token blocked
    with probability 1/100).  A state with no valid token is given one random token.
    """
    kinds = rng.integers(0, 3, size=positions)
    out = np.zeros((positions, V), dtype=bool)
    for i, k in enumerate(kinds):
        if k == 0:
            out[i, rng.choice(V, size=min(64, V), replace=False)] = True
        elif k == 1:
            out[i] = rng.random(V) < 0.5
        else:
            out[i] = rng.random(V) >= 0.01
        if not out[i].any():
            out[i, rng.integers(0, V)] = True
    return out


def pack_valid_sets(valid: np.ndarray) -> np.ndarray:
    """bool [..., V] -> uint32 words [..., ceil(V/32)]: bit v % 32 of word v // 32 = valid[..., v]."""
    V = valid.shape[-1]
    W = (V + 31) // 32
    pad = np.zeros(valid.shape[:-1] + (W * 32,), dtype=bool)
    pad[..., :V] = valid
    by = np.packbits(pad, axis=-1, bitorder="little")
    return np.ascontiguousarray(by).view("<u4").astype(np.uint32)


def unpack_valid_sets(words: np.ndarray, V: int) -> np.ndarray:
    """Inverse of pack_valid_sets."""
    by = np.ascontiguousarray(words, dtype="<u4").view(np.uint8)
    return np.unpackbits(by, axis=-1, bitorder="little")[..., :V].astype(bool)


def draft_nucleus_mask(x: np.ndarray, temperature: float, top_p: float) -> np.ndarray | None:
    """The draft sampler's own top-p set per row of stored logits x [..., V]: the tokens of largest
    logit, whole groups of equal logit at a time, until the mass of softmax(x / T) they hold first
    reaches top_p (the proposal side's processor, so that draft tokens are draws from it)."""
    if not top_p < 1.0:
        return None
    flat = x.reshape(-1, x.shape[-1])
    keep = np.zeros(flat.shape, dtype=bool)
    for r, row in enumerate(flat):
        z = row / temperature
        w = np.exp(z - z.max())
        w /= w.sum()
        vals, inv = np.unique(row, return_inverse=True)       # ascending distinct logits
        mass = np.bincount(inv, weights=w, minlength=vals.size)[::-1]  # descending
        cum = np.cumsum(mass)
        j = int(np.searchsorted(cum, top_p, side="left"))
        g = vals[::-1][min(j, vals.size - 1)]
        keep[r] = row >= g
    return keep.reshape(x.shape)


def _nthreads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


# ------------------------------------------------------------------ spec-verify batches

@dataclass
class SpecBatch:
    cfg: SpecConfig
    target: np.ndarray       # [B, gamma+1, V] uint16 (bf16 bits) or float32
    draft: np.ndarray        # [B, gamma,   V]
    draft_tokens: np.ndarray  # [B, gamma] int32
    uniforms: np.ndarray     # [B, gamma+2] float32
    meta: dict = field(default_factory=dict)
    allowed: np.ndarray | None = None  # grammar mask words [B, gamma+1, ceil(V/32)] uint32

    @property
    def rows(self) -> int:
        return self.cfg.B * (2 * self.cfg.gamma + 1)

    @property
    def logit_bytes(self) -> int:
        return self.target.nbytes + self.draft.nbytes


def make_spec_batch(cfg: SpecConfig, *, threads: int | None = None) -> SpecBatch:
    B, g, V = cfg.B, cfg.gamma, cfg.V
    ss_logit, ss_draw, ss_unif = np.random.SeedSequence(cfg.seed).spawn(3)
    req_logit = ss_logit.spawn(B)
    req_draw = ss_draw.spawn(B)
    req_unif = ss_unif.spawn(B)
    bias = _zipf_bias(V, cfg.seed) if cfg.target == "zipf" else None
    sdt = np.uint16 if cfg.dtype == "bf16" else np.float32
    target = np.empty((B, g + 1, V), dtype=sdt)
    draft = np.empty((B, g, V), dtype=sdt)
    tokens = np.empty((B, g), dtype=np.int32)
    uniforms = np.empty((B, g + 2), dtype=np.float32)
    allowed = np.empty((B, g + 1, (V + 31) // 32), dtype=np.uint32) if cfg.mask else None
    req_mask = np.random.SeedSequence([cfg.seed, 11]).spawn(B) if cfg.mask else None

    def one(b):
        rng = np.random.Generator(np.random.PCG64(req_logit[b]))
        t32 = _target_rows(rng, cfg.target, g + 1, V, bias)
        d32 = (cfg.draft_scale * t32[:g].astype(np.float64)
               + rng.standard_normal((g, V)) * cfg.draft_noise).astype(np.float32)
        target[b] = _store(t32, cfg.dtype)
        draft[b] = _store(d32, cfg.dtype)
        xd = stored_to_f64(draft[b])
        keep = draft_keep_mask(xd, cfg.top_k)
        if cfg.top_p < 1.0:
            keep = draft_nucleus_mask(xd, cfg.temperature, cfg.top_p)
        if cfg.mask:
            valid = grammar_valid_sets(np.random.Generator(np.random.PCG64(req_mask[b])), g + 1, V)
            allowed[b] = pack_valid_sets(valid)
            keep = valid[:g] if keep is None else keep & valid[:g]
        tokens[b] = gumbel_max_tokens(np.random.Generator(np.random.PCG64(req_draw[b])),
                                      xd / cfg.temperature, keep)
        uniforms[b] = uniforms_from(np.random.Generator(np.random.PCG64(req_unif[b])), g + 2)

    n = threads or _nthreads()
    if n > 1 and B > 1:
        with ThreadPoolExecutor(n) as ex:
            list(ex.map(one, range(B)))
    else:
        for b in range(B):
            one(b)
    return SpecBatch(cfg, target, draft, tokens, uniforms, allowed=allowed)


def redraw(batch: SpecBatch, trial_seed: int) -> SpecBatch:
    """Same logits, fresh draft tokens and uniforms (the c1 trial recipe)."""
    cfg = batch.cfg
    ss_draw, ss_unif = np.random.SeedSequence([cfg.seed, trial_seed]).spawn(2)
    B = cfg.B
    tokens = np.empty_like(batch.draft_tokens)
    unif = np.empty_like(batch.uniforms)
    for b in range(B):
        xd = stored_to_f64(batch.draft[b])
        keep = draft_keep_mask(xd, cfg.top_k)
        tokens[b] = gumbel_max_tokens(np.random.Generator(np.random.PCG64(ss_draw.spawn(B)[b])),
                                      xd / cfg.temperature, keep)
        unif[b] = uniforms_from(np.random.Generator(np.random.PCG64(ss_unif.spawn(B)[b])),
                                cfg.gamma + 2)
    return SpecBatch(cfg, batch.target, batch.draft, tokens, unif, dict(batch.meta, trial=trial_seed))


def trial_batches(cfg: SpecConfig, trials: int, *, redraw_logits: bool = False):
    """``trials`` independent single-config draws stacked along the request axis.

    With ``redraw_logits`` False the logits of request 0 are repeated and only draft tokens and
    uniforms change per trial; with True every trial draws its own logits too.
    """
    if redraw_logits:
        return make_spec_batch(scaled(cfg, B=trials))
    base = make_spec_batch(scaled(cfg, B=1))
    g, V = cfg.gamma, cfg.V
    target = np.broadcast_to(base.target, (trials, g + 1, V)).copy()
    draft = np.broadcast_to(base.draft, (trials, g, V)).copy()
    ss_draw, ss_unif = np.random.SeedSequence([cfg.seed, 99]).spawn(2)
    rng_d = np.random.Generator(np.random.PCG64(ss_draw))
    rng_u = np.random.Generator(np.random.PCG64(ss_unif))
    xd = stored_to_f64(base.draft[0])
    keep = draft_keep_mask(xd, cfg.top_k)
    z = xd / cfg.temperature
    tokens = np.stack([gumbel_max_tokens(rng_d, z, keep) for _ in range(trials)]).astype(np.int32)
    unif = uniforms_from(rng_u, (trials, g + 2))
    return SpecBatch(scaled(cfg, B=trials), target, draft, tokens, unif, dict(trials=trials))


# ------------------------------------------------------------------ trees

def medusa_tree_parents(branching, max_nodes: int | None = None) -> np.ndarray:
    """Parent array of a Cartesian candidate tree in BFS order.

    Level 1 has branching[0] nodes (parent -1); every node of level d has branching[d] children.
    Truncating the BFS order keeps the tree ancestor-closed.
    """
    parents = []
    level = [-1]
    for w in branching:
        nxt = []
        for p in level:
            for _ in range(w):
                parents.append(p)
                nxt.append(len(parents) - 1)
        level = nxt
    par = np.array(parents, dtype=np.int32)
    return par if max_nodes is None else par[:max_nodes]


@dataclass
class TreeBatch:
    cfg: TreeConfig
    logits: np.ndarray    # [B, N+1, V]
    parents: np.ndarray   # [B, N] int32
    tokens: np.ndarray    # [B, N] int32
    meta: dict = field(default_factory=dict)
    uniforms: np.ndarray | None = None  # [B] float32: typical acceptance's final draw

    @property
    def rows(self) -> int:
        return self.logits.shape[0] * self.logits.shape[1]

    @property
    def logit_bytes(self) -> int:
        return self.logits.nbytes


def make_tree_batch(cfg: TreeConfig, *, threads: int | None = None) -> TreeBatch:
    """Tree logits drawn like c3's target; node tokens copy the predictor row's argmax with
    probability p_match (the draft heads' stand-in), else a uniform token."""
    par = medusa_tree_parents(cfg.branching, cfg.max_nodes)
    N, B, V = len(par), cfg.B, cfg.V
    ss_logit, ss_tok = np.random.SeedSequence(cfg.seed).spawn(2)
    req_logit, req_tok = ss_logit.spawn(B), ss_tok.spawn(B)
    bias = _zipf_bias(V, cfg.seed)
    sdt = np.uint16 if cfg.dtype == "bf16" else np.float32
    logits = np.empty((B, N + 1, V), dtype=sdt)
    tokens = np.empty((B, N), dtype=np.int32)

    def one(b):
        rng = np.random.Generator(np.random.PCG64(req_logit[b]))
        logits[b] = _store(_target_rows(rng, "zipf", N + 1, V, bias), cfg.dtype)
        top = np.argmax(stored_to_f64(logits[b]), axis=-1)  # first index of the maximum
        r2 = np.random.Generator(np.random.PCG64(req_tok[b]))
        match = r2.random(N) < cfg.p_match
        rand = r2.integers(0, V, size=N)
        pred = np.where(par < 0, 0, par + 1)
        tokens[b] = np.where(match, top[pred], rand).astype(np.int32)

    n = threads or _nthreads()
    if n > 1 and B > 1:
        with ThreadPoolExecutor(n) as ex:
            list(ex.map(one, range(B)))
    else:
        for b in range(B):
            one(b)
    unif = None
    if cfg.typical:
        unif = uniforms_from(np.random.Generator(np.random.PCG64(
            np.random.SeedSequence([cfg.seed, 13]))), B)
    return TreeBatch(cfg, logits, np.broadcast_to(par, (B, N)).copy(), tokens, uniforms=unif)


# ------------------------------------------------------------------ sampled trees

@dataclass
class SampleTreeBatch:
    cfg: SampleTreeConfig
    target: np.ndarray    # [B, N+1, V]
    draft: np.ndarray     # [B, N+1, V]: row 0 frontier, row i+1 at node i
    parents: np.ndarray   # [B, N] int32
    tokens: np.ndarray    # [B, N] int32
    qrow: np.ndarray      # [B, N] int32 = parent + 1
    uniforms: np.ndarray  # [B, N+1] float32
    meta: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return self.target.shape[0] * self.target.shape[1]


def make_sample_tree_batch(cfg: SampleTreeConfig, *, parents=None,
                           threads: int | None = None) -> SampleTreeBatch:
    """Target rows as c3's target, draft rows 0.8 * target + noise; each node's token a Gumbel-max
    draw from softmax(draft row at its parent / T) (the drafter's own sampler, outside the verify
    step), so the children of one node are i.i.d. given their parent."""
    par = medusa_tree_parents(cfg.branching, cfg.max_nodes) if parents is None else \
        np.asarray(parents, dtype=np.int32)
    N, B, V = len(par), cfg.B, cfg.V
    ss_logit, ss_draw, ss_unif = np.random.SeedSequence(cfg.seed).spawn(3)
    req_logit, req_draw, req_unif = ss_logit.spawn(B), ss_draw.spawn(B), ss_unif.spawn(B)
    bias = _zipf_bias(V, cfg.seed)
    sdt = np.uint16 if cfg.dtype == "bf16" else np.float32
    target = np.empty((B, N + 1, V), dtype=sdt)
    draft = np.empty((B, N + 1, V), dtype=sdt)
    tokens = np.empty((B, N), dtype=np.int32)
    uniforms = np.empty((B, N + 1), dtype=np.float32)
    qrow = (par + 1).astype(np.int32)

    def one(b):
        rng = np.random.Generator(np.random.PCG64(req_logit[b]))
        t32 = _target_rows(rng, "zipf", N + 1, V, bias)
        d32 = (cfg.draft_scale * t32.astype(np.float64)
               + rng.standard_normal((N + 1, V)) * cfg.draft_noise).astype(np.float32)
        target[b] = _store(t32, cfg.dtype)
        draft[b] = _store(d32, cfg.dtype)
        if N:
            z = stored_to_f64(draft[b][qrow]) / cfg.temperature
            tokens[b] = gumbel_max_tokens(np.random.Generator(np.random.PCG64(req_draw[b])), z)
        uniforms[b] = uniforms_from(np.random.Generator(np.random.PCG64(req_unif[b])), N + 1)

    n = threads or _nthreads()
    if n > 1 and B > 1:
        with ThreadPoolExecutor(n) as ex:
            list(ex.map(one, range(B)))
    else:
        for b in range(B):
            one(b)
    return SampleTreeBatch(cfg, target, draft, np.broadcast_to(par, (B, N)).copy(), tokens,
                           np.broadcast_to(qrow, (B, N)).copy(), uniforms)


# ------------------------------------------------------------------ SMC-SD rounds

@dataclass
class SmcBatch:
    cfg: SmcConfig
    target: np.ndarray    # [B, K+1, V]
    draft: np.ndarray     # [B, K, V]
    draft_tokens: np.ndarray  # [B, K] int32
    log_weights: np.ndarray   # [B] float32
    uniforms: np.ndarray  # [B, 2] float32
    meta: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return self.cfg.B * (2 * self.cfg.K + 1)

    @property
    def logit_bytes(self) -> int:
        return self.target.nbytes + self.draft.nbytes


def make_smc_batch(cfg: SmcConfig, *, threads: int | None = None) -> SmcBatch:
    """Particles drawn like c3's requests: target rows N(0,3^2) + Zipf bias, draft rows
    0.8 * target + noise, draft tokens Gumbel-max draws from q (the drafter's sampler, outside the
    verify step); incoming log weights N(0, logw_sd^2); uniforms for the extension and the ancestor."""
    B, K, V = cfg.B, cfg.K, cfg.V
    ss_logit, ss_draw, ss_unif = np.random.SeedSequence(cfg.seed).spawn(3)
    req_logit, req_draw, req_unif = ss_logit.spawn(B), ss_draw.spawn(B), ss_unif.spawn(B)
    bias = _zipf_bias(V, cfg.seed)
    sdt = np.uint16 if cfg.dtype == "bf16" else np.float32
    target = np.empty((B, K + 1, V), dtype=sdt)
    draft = np.empty((B, K, V), dtype=sdt)
    tokens = np.empty((B, K), dtype=np.int32)
    uniforms = np.empty((B, 2), dtype=np.float32)
    logw = np.empty(B, dtype=np.float32)

    def one(b):
        rng = np.random.Generator(np.random.PCG64(req_logit[b]))
        t32 = _target_rows(rng, "zipf", K + 1, V, bias)
        d32 = (cfg.draft_scale * t32[:K].astype(np.float64)
               + rng.standard_normal((K, V)) * cfg.draft_noise).astype(np.float32)
        target[b] = _store(t32, cfg.dtype)
        draft[b] = _store(d32, cfg.dtype)
        r2 = np.random.Generator(np.random.PCG64(req_draw[b]))
        if K:
            tokens[b] = gumbel_max_tokens(r2, stored_to_f64(draft[b]) / cfg.temperature)
        logw[b] = np.float32(r2.standard_normal() * cfg.logw_sd)
        uniforms[b] = uniforms_from(np.random.Generator(np.random.PCG64(req_unif[b])), 2)

    n = threads or _nthreads()
    if n > 1 and B > 1:
        with ThreadPoolExecutor(n) as ex:
            list(ex.map(one, range(B)))
    else:
        for b in range(B):
            one(b)
    return SmcBatch(cfg, target, draft, tokens, logw, uniforms)
