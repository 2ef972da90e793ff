"""Seeded synthetic inputs for paged-KV attention.

This module only draws data: sequence lengths, page permutations, N(0,1)
values rounded to bf16, and (for the fp8 cache) per-page e4m3 codes with their
fp32 scales.  It holds none of the attention arithmetic, and it is the one
module that both the oracle-side tests and the CUDA-side tests/bench use.

Workloads follow the call shapes of the pages:

* decode step: ``groups`` sequences x ``rows`` = 1 ("kern manifest v7",
  $defs.Batch, e.g. {"groups": 256, "rows": 1});
* speculative verify round: ``rows`` = 8, causal within the round
  ($defs.Batch `rows`: "8 for a speculative round -- exact, not a bound");
* prefill chunk: ``groups`` = 1, ``rows`` = the chunk's tokens, over a longer
  cached context ($defs.Batch `context`).

Recipe (all draws from numpy PCG64, seeded):

* SeedSequence(seed).spawn(4) gives four streams: lengths + page permutation,
  Q, K, V.  K and V are drawn in fixed-size chunks, each from its own spawned
  child stream, so the values do not depend on the thread count.
* values ~ N(0, 1) in float32, rounded to bf16 (round-to-nearest-even, by
  torch's CPU conversion).
* fp8 cache: per physical page and per pool, scale = amax(|x|) / 448 (1 when
  amax is 0), code = e4m3fn(round-to-nearest-even(x / scale)) (torch's CPU
  conversion), so value = code * scale.
* the pool holds exactly the pages the sequences need (the tiny case: 64), in
  a random permutation; page-table entries past a sequence's last page are -1.
* ``poison=True`` fills every token slot past a sequence's length, and every
  unreferenced page, with NaN codes, so any read of them shows in the output.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np
import torch

KV_BF16 = 0
KV_FP8_E4M3 = 1

BF16_NAN = 0x7FC0
E4M3_NAN = 0x7F
E4M3_MAX = 448.0

_CHUNK_ELEMS = 1 << 22


@dataclass(frozen=True)
class Config:
    name: str
    groups: int
    rows: int
    n_head: int
    n_head_kv: int
    head_dim: int
    page_size: int
    kv_dtype: int
    seed: int
    lens: str                 # how seq_lens are drawn
    pages_per_seq: int        # page-table row stride (capacity in pages)
    pool_pages: int | None = None   # None: exactly the pages the sequences need
    meta: dict = field(default_factory=dict)
    # Ragged rows: "NxR,..." gives N sequences of R rows each, in call order
    # (a mixed step: decode rows, verify rounds and prefill chunks side by
    # side); `rows` is then the largest R.  None: every sequence has `rows`.
    q_lens: str | None = None
    # Draft-tree rows: each sequence's rows are a random forest of proposals
    # flattened parents-first, given to the op as one mask word per row.
    tree: bool = False

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.head_dim)))


# The five workloads.  `meta` mirrors the model metadata a caller reads
# head_dim from ("Radiance architecture plugins", section "Declare: the
# metadata": head_dim is read, never derived; on the hybrids hidden/heads
# is 213 while head_dim is 256).
CONFIGS: dict[str, Config] = {
    "tiny_decode": Config("tiny_decode", 4, 1, 8, 2, 128, 16, KV_BF16, 0, "fixed:37,64,129,300",
                          pages_per_seq=19, pool_pages=64,
                          meta=dict(n_head=8, n_head_kv=2, head_dim=128, n_embd=1024)),
    "batched_decode": Config("batched_decode", 256, 1, 32, 8, 128, 16, KV_BF16, 1, "uniform:512,8192",
                             pages_per_seq=512,
                             meta=dict(n_head=32, n_head_kv=8, head_dim=128, n_embd=4096)),
    "hybrid_decode": Config("hybrid_decode", 128, 1, 16, 2, 256, 32, KV_BF16, 2,
                            "loguniform:1024,32768", pages_per_seq=1024,
                            meta=dict(n_head=16, n_head_kv=2, head_dim=256, n_embd=3408)),
    "spec_verify": Config("spec_verify", 64, 8, 32, 8, 128, 16, KV_FP8_E4M3, 3, "uniform:2048,16384",
                          pages_per_seq=1024,
                          meta=dict(n_head=32, n_head_kv=8, head_dim=128, n_embd=4096)),
    "prefill_chunk": Config("prefill_chunk", 1, 2048, 32, 8, 128, 16, KV_BF16, 4, "fixed:8192",
                            pages_per_seq=512, pool_pages=512,
                            meta=dict(n_head=32, n_head_kv=8, head_dim=128, n_embd=4096)),
    # The prefill chunk over fp8-e4m3 pools (per-page scales).
    "prefill_chunk_fp8": Config("prefill_chunk_fp8", 1, 2048, 32, 8, 128, 16, KV_FP8_E4M3, 7, "fixed:8192",
                                pages_per_seq=512, pool_pages=512,
                                meta=dict(n_head=32, n_head_kv=8, head_dim=128, n_embd=4096)),
    # The verify round as a draft tree of 8 proposals per sequence instead of
    # a chain ("Radiance architecture plugins", section "Declare: drafters,
    # encoders, generators": rad_drafter_tree).
    "tree_verify": Config("tree_verify", 64, 8, 32, 8, 128, 16, KV_FP8_E4M3, 5, "uniform:2048,16384",
                          pages_per_seq=1024, tree=True,
                          meta=dict(n_head=32, n_head_kv=8, head_dim=128, n_embd=4096)),
    # A continuous-batching step ("Radiance architecture plugins", section
    # "Step: issuing the graph": a prefill chunk beside decode rows, decode
    # first): 96 decode rows, 24 verify rounds of 8 and one 256-row chunk.
    "mixed_step": Config("mixed_step", 121, 256, 32, 8, 128, 16, KV_BF16, 6, "uniform:512,8192",
                         pages_per_seq=512, q_lens="96x1,24x8,1x256",
                         meta=dict(n_head=32, n_head_kv=8, head_dim=128, n_embd=4096)),
    # The hybrid model's shapes at head_dim 256 (read from its metadata): its
    # decode over an fp8 cache, and a prefill chunk over bf16 and fp8 caches.
    "hybrid_decode_fp8": Config("hybrid_decode_fp8", 128, 1, 16, 2, 256, 32, KV_FP8_E4M3, 8,
                                "loguniform:1024,32768", pages_per_seq=1024,
                                meta=dict(n_head=16, n_head_kv=2, head_dim=256, n_embd=3408)),
    "prefill_chunk_d256": Config("prefill_chunk_d256", 1, 2048, 16, 2, 256, 32, KV_BF16, 9, "fixed:8192",
                                 pages_per_seq=256, pool_pages=256,
                                 meta=dict(n_head=16, n_head_kv=2, head_dim=256, n_embd=3408)),
    "prefill_chunk_d256_fp8": Config("prefill_chunk_d256_fp8", 1, 2048, 16, 2, 256, 32, KV_FP8_E4M3, 10,
                                     "fixed:8192", pages_per_seq=256, pool_pages=256,
                                     meta=dict(n_head=16, n_head_kv=2, head_dim=256, n_embd=3408)),
}


@dataclass
class Workload:
    cfg: Config
    q: np.ndarray            # uint16 bf16 bits [G, R, H, D]; ragged: [T, H, D] packed by q_lens
    k_pool: np.ndarray       # uint16 or uint8 [num_pages, P, Hkv, D]
    v_pool: np.ndarray
    page_table: np.ndarray   # int32 [G, pages_per_seq]
    seq_lens: np.ndarray     # int32 [G]
    k_scales: np.ndarray | None   # float32 [num_pages] (fp8 only)
    v_scales: np.ndarray | None
    q_lens: np.ndarray | None = None     # int32 [G] rows per sequence (ragged calls)
    tree_mask: np.ndarray | None = None  # uint32 [G, R] path bits per row (tree calls)

    @property
    def ragged(self) -> bool:
        return self.q_lens is not None

    def rows_of(self) -> np.ndarray:
        """Rows of every sequence (int64 [G])."""
        if self.q_lens is None:
            return np.full(self.groups, self.cfg.rows, dtype=np.int64)
        return self.q_lens.astype(np.int64)

    def packed(self):
        """The op's ragged inputs: q [T, H, D] with sequence g's rows at
        cu[g] .. cu[g+1]-1, cu int32 [G + 1], and the mask words of those rows
        (or None)."""
        ql = self.rows_of()
        cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
        q = self.q if self.ragged else self.q.reshape(-1, *self.q.shape[2:])
        mask = None
        if self.tree_mask is not None:
            mask = np.concatenate([self.tree_mask[g, :ql[g]] for g in range(self.groups)])
        return np.ascontiguousarray(q), cu, mask

    @property
    def groups(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def pages_per_seq(self) -> int:
        return int(self.page_table.shape[1])

    def call_args(self) -> dict:
        c = self.cfg
        return dict(rows=c.rows, n_head=c.n_head, n_head_kv=c.n_head_kv, head_dim=c.head_dim,
                    page_size=c.page_size, scale=c.scale, kv_dtype=c.kv_dtype)

    def select_groups(self, idx) -> "Workload":
        """The same pool, with only the listed sequences (in that order) in the call."""
        idx = np.asarray(idx, dtype=np.int64)
        if self.ragged:
            _, cu, _ = self.packed()
            q = np.concatenate([self.q[cu[g]:cu[g + 1]] for g in idx], axis=0)
        else:
            q = self.q[idx]
        return replace(self, q=np.ascontiguousarray(q),
                       page_table=np.ascontiguousarray(self.page_table[idx]),
                       seq_lens=np.ascontiguousarray(self.seq_lens[idx]),
                       q_lens=None if self.q_lens is None else np.ascontiguousarray(self.q_lens[idx]),
                       tree_mask=None if self.tree_mask is None else np.ascontiguousarray(self.tree_mask[idx]))


def compact_pool(w: Workload) -> Workload:
    """The same call over a pool holding only the pages its sequences use
    (page ids renumbered in pool order), e.g. after select_groups."""
    used = np.unique(w.page_table[w.page_table >= 0])
    remap = np.full(w.num_pages, -1, dtype=np.int32)
    remap[used] = np.arange(used.size, dtype=np.int32)
    table = np.where(w.page_table >= 0, remap[np.maximum(w.page_table, 0)], -1).astype(np.int32)
    sc = (lambda a: None if a is None else np.ascontiguousarray(a[used]))
    return replace(w, k_pool=np.ascontiguousarray(w.k_pool[used]), v_pool=np.ascontiguousarray(w.v_pool[used]),
                   page_table=table, k_scales=sc(w.k_scales), v_scales=sc(w.v_scales))


# ---------------------------------------------------------------- draft trees
# A draft tree of R proposals is flattened parents-first: parents[r] < r, or
# -1 for a node hanging directly off the cached context.  The op takes one
# mask word per node with bit i set for every node i on the node's path.

def path_of(parents, r):
    """Nodes from r up to the cached context, r first."""
    path = []
    while r >= 0:
        path.append(r)
        r = parents[r]
    return path


def mask_words(parents):
    """Tree-mask word of every node: bit i for each node on its path."""
    return np.array([sum(1 << i for i in path_of(parents, r)) for r in range(len(parents))],
                    dtype=np.uint32)


def random_parents(rng, R, forest=True):
    lo = -1 if forest else 0
    return [-1] + [int(rng.integers(lo, r)) for r in range(1, R)]


def chain(R):
    return list(range(-1, R - 1))


def parse_q_lens(spec: str) -> list[int]:
    out = []
    for part in spec.split(","):
        n, r = part.split("x")
        out += [int(r)] * int(n)
    return out


def draw_seq_lens(cfg: Config, rng: np.random.Generator) -> np.ndarray:
    kind, arg = cfg.lens.split(":")
    if kind == "fixed":
        vals = [int(x) for x in arg.split(",")]
        out = np.array(vals if len(vals) == cfg.groups else vals * cfg.groups, dtype=np.int64)[: cfg.groups]
    elif kind == "uniform":
        lo, hi = (int(x) for x in arg.split(","))
        out = rng.integers(lo, hi, size=cfg.groups, endpoint=True)
    elif kind == "loguniform":
        lo, hi = (int(x) for x in arg.split(","))
        out = np.rint(np.exp(rng.uniform(math.log(lo), math.log(hi), size=cfg.groups))).astype(np.int64)
    else:
        raise ValueError(cfg.lens)
    return out.astype(np.int32)


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def _quantise_e4m3_pages(x: np.ndarray):
    """x float32 [pages, ...] -> (uint8 codes, float32 per-page scales)."""
    pages = x.shape[0]
    amax = np.abs(x.reshape(pages, -1)).max(axis=1)
    scales = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    y = torch.from_numpy(x / scales.reshape((pages,) + (1,) * (x.ndim - 1)))
    codes = y.clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes, scales


def _fill_pool(ss: np.random.SeedSequence, num_pages: int, page_elems: int, kv_dtype: int,
               threads: int):
    pages_per_chunk = max(1, _CHUNK_ELEMS // page_elems)
    n_chunks = (num_pages + pages_per_chunk - 1) // pages_per_chunk
    children = ss.spawn(n_chunks)
    dt = np.uint16 if kv_dtype == KV_BF16 else np.uint8
    pool = np.empty((num_pages, page_elems), dtype=dt)
    scales = np.empty(num_pages, dtype=np.float32) if kv_dtype == KV_FP8_E4M3 else None

    def work(i):
        p0 = i * pages_per_chunk
        p1 = min(num_pages, p0 + pages_per_chunk)
        x = np.random.Generator(np.random.PCG64(children[i])).standard_normal(
            (p1 - p0, page_elems), dtype=np.float32)
        if kv_dtype == KV_BF16:
            pool[p0:p1] = _f32_to_bf16_bits(x)
        else:
            codes, sc = _quantise_e4m3_pages(x)
            pool[p0:p1] = codes
            scales[p0:p1] = sc

    with ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
        list(ex.map(work, range(n_chunks)))
    return pool, scales


def make_workload(cfg: Config | str, *, poison: bool = False, threads: int | None = None) -> Workload:
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    threads = threads or min(16, (torch.get_num_threads() or 1))
    ss_meta, ss_q, ss_k, ss_v = np.random.SeedSequence(cfg.seed).spawn(4)
    rng = np.random.Generator(np.random.PCG64(ss_meta))
    seq_lens = draw_seq_lens(cfg, rng)
    q_lens = None
    if cfg.q_lens is not None:
        q_lens = np.array(parse_q_lens(cfg.q_lens), dtype=np.int32)
        assert q_lens.shape == (cfg.groups,) and int(q_lens.max()) == cfg.rows
        seq_lens = np.maximum(seq_lens, q_lens)
    P = cfg.page_size
    n_pages_seq = (seq_lens.astype(np.int64) + P - 1) // P
    assert int(n_pages_seq.max()) <= cfg.pages_per_seq
    need = int(n_pages_seq.sum())
    num_pages = cfg.pool_pages if cfg.pool_pages is not None else need
    assert num_pages >= need
    perm = rng.permutation(num_pages).astype(np.int32)
    page_table = np.full((cfg.groups, cfg.pages_per_seq), -1, dtype=np.int32)
    off = 0
    for g in range(cfg.groups):
        n = int(n_pages_seq[g])
        page_table[g, :n] = perm[off:off + n]
        off += n

    q_shape = ((int(q_lens.sum()),) if q_lens is not None else (cfg.groups, cfg.rows)) + (cfg.n_head, cfg.head_dim)
    q32 = np.random.Generator(np.random.PCG64(ss_q)).standard_normal(q_shape, dtype=np.float32)
    q = _f32_to_bf16_bits(q32)
    page_elems = P * cfg.n_head_kv * cfg.head_dim
    k_flat, k_scales = _fill_pool(ss_k, num_pages, page_elems, cfg.kv_dtype, threads)
    v_flat, v_scales = _fill_pool(ss_v, num_pages, page_elems, cfg.kv_dtype, threads)
    shape = (num_pages, P, cfg.n_head_kv, cfg.head_dim)
    tree_mask = None
    if cfg.tree:
        assert cfg.rows <= 32
        tree_mask = np.zeros((cfg.groups, cfg.rows), dtype=np.uint32)
        for g in range(cfg.groups):
            n = cfg.rows if q_lens is None else int(q_lens[g])
            tree_mask[g, :n] = mask_words(random_parents(rng, n)) if n else []
    w = Workload(cfg, q, k_flat.reshape(shape), v_flat.reshape(shape), page_table, seq_lens,
                 k_scales, v_scales, q_lens, tree_mask)
    if poison:
        poison_unused(w)
    return w


def poison_unused(w: Workload) -> None:
    """NaN codes in every token slot no sequence of the call may read."""
    nan = BF16_NAN if w.cfg.kv_dtype == KV_BF16 else E4M3_NAN
    P = w.cfg.page_size
    used = np.zeros(w.num_pages, dtype=bool)
    for g in range(w.groups):
        L = int(w.seq_lens[g])
        n = (L + P - 1) // P
        pages = w.page_table[g, :n]
        used[pages] = True
        tail = L - (n - 1) * P
        if tail < P:
            last = pages[n - 1]
            w.k_pool[last, tail:] = nan
            w.v_pool[last, tail:] = nan
    w.k_pool[~used] = nan
    w.v_pool[~used] = nan


def kv_bytes(w: Workload) -> int:
    """Algorithmic KV bytes of one call: every visible key's K and V row for
    every KV head, the per-page scales (fp8) and the page-table entries read."""
    c = w.cfg
    e = 2 if c.kv_dtype == KV_BF16 else 1
    # a sequence with rows reads every key (its last row, or with a tree each
    # node its own key, sees them); one without rows reads nothing
    L = np.where(w.rows_of() > 0, w.seq_lens.astype(np.int64), 0)
    pages = (L + c.page_size - 1) // c.page_size
    b = int(L.sum()) * c.n_head_kv * c.head_dim * 2 * e
    if c.kv_dtype == KV_FP8_E4M3:
        b += int(pages.sum()) * 2 * 4
    b += int(pages.sum()) * 4
    return b


def aux_bytes(w: Workload) -> int:
    """Q read, output written and seq_lens read by one call."""
    c = w.cfg
    b = 2 * int(w.rows_of().sum()) * c.n_head * c.head_dim * 2 + 4 * w.groups
    if w.ragged:
        b += 4 * (w.groups + 1)
    if w.tree_mask is not None:
        b += 4 * int(w.rows_of().sum())
    return b


def attended_flops(w: Workload) -> int:
    """4*D flops (QK and PV multiply-adds) per visible (row, head, key)."""
    c = w.cfg
    L = w.seq_lens.astype(np.int64)
    R = w.rows_of()
    keys = 0
    for g in range(w.groups):
        for r in range(int(R[g])):
            if w.tree_mask is not None:
                keys += int(L[g] - R[g]) + bin(int(w.tree_mask[g, r])).count("1")
            else:
                keys += int(L[g] - R[g] + r + 1)
    return keys * c.n_head * 4 * c.head_dim
