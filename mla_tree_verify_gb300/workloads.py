"""Seeded synthetic inputs for MLA tree-verify attention.

This module only draws inputs: request sizes, scattered page_size=1 slots, draft
trees, the flattened custom mask and bf16 tensors.  It holds none of the attention
arithmetic, so both the CUDA path and the fp64 oracle can use it.

Layouts (all arrays are numpy, C-contiguous):

* ``q``            uint16 (bf16 bits) ``[total_q, H, 576]``
* ``kv_cache``     uint16 (bf16 bits) ``[num_slots, 576]``; the first 512 dims are the
  latent (also V), the last 64 the rope part.  Slots that no request references hold
  bf16 NaN, so a stray gather shows up in the output.
* ``kv_indices``   int32 ``[kv_indptr[bs]]`` prefix slots, request after request.
* ``kv_indptr``    int32 ``[bs+1]`` (prefix lengths P_b).
* ``out_cache_loc`` int64 ``[total_q]`` slot of each draft token's own KV row.
* ``qo_indptr``    int64 ``[bs+1]`` (draft counts T_b).
* ``custom_mask``  uint8 ``[sum_b T_b*(P_b+T_b)]``: per request a row-major
  ``[T_b, P_b+T_b]`` block; prefix columns are 1, draft column j is 1 in row i iff
  j is an ancestor of i or j == i.
* ``mask_indptr``  int64 ``[bs+1]`` offsets of those blocks.

Draft trees are topologically ordered (parent < child): a random tree draws
``parent[i]`` uniformly from ``[0, i)``, a chain uses ``parent[i] = i-1``.
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np

HEADS = 64
D_QK = 576
D_V = 512
BF16_NAN = np.uint16(0x7FC0)
NSPLIT = 64
SM_SCALE = 1.0 / math.sqrt(192.0)


@dataclasses.dataclass
class Workload:
    name: str
    q: np.ndarray
    kv_cache: np.ndarray
    kv_indices: np.ndarray
    kv_indptr: np.ndarray
    out_cache_loc: np.ndarray
    custom_mask: np.ndarray
    mask_indptr: np.ndarray
    qo_indptr: np.ndarray
    parents: list  # per request: int64 array of parent ids (-1 for the root)
    sm_scale: float = SM_SCALE

    @property
    def bs(self) -> int:
        return int(self.kv_indptr.shape[0] - 1)

    @property
    def num_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_slots(self) -> int:
        return int(self.kv_cache.shape[0])

    @property
    def prefix_lens(self) -> np.ndarray:
        return np.diff(self.kv_indptr.astype(np.int64))

    @property
    def draft_lens(self) -> np.ndarray:
        return np.diff(self.qo_indptr)

    @property
    def max_q_per_req(self) -> int:
        return int(self.draft_lens.max()) if self.bs else 0

    def visible_pairs(self) -> int:
        """Number of visible (query token, key column) pairs, per head."""
        n = 0
        for b in range(self.bs):
            P = int(self.prefix_lens[b])
            T = int(self.draft_lens[b])
            blk = self.mask_block(b)
            n += T * P + int(blk[:, P:].astype(bool).sum())
        return n

    def mask_block(self, b: int) -> np.ndarray:
        P = int(self.prefix_lens[b])
        T = int(self.draft_lens[b])
        s = int(self.mask_indptr[b])
        return self.custom_mask[s:s + T * (P + T)].reshape(T, P + T)

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes: every referenced row (prefix + drafts) read once."""
        return int((self.prefix_lens.sum() + self.draft_lens.sum()) * D_QK * 2)


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_float32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(seed_seq: np.random.SeedSequence, n_rows: int, width: int,
                 chunk_rows: int = 65536, threads: int = 8) -> np.ndarray:
    """N(0,1) bf16 bits [n_rows, width], drawn chunk by chunk from spawned seeds so
    the values do not depend on the thread count."""
    out = np.empty((n_rows, width), dtype=np.uint16)
    n_chunks = max(1, (n_rows + chunk_rows - 1) // chunk_rows)
    children = seed_seq.spawn(n_chunks)

    def work(k):
        lo = k * chunk_rows
        hi = min(n_rows, lo + chunk_rows)
        if hi <= lo:
            return
        g = np.random.default_rng(children[k])
        out[lo:hi] = _bf16_bits(g.standard_normal((hi - lo, width), dtype=np.float32))

    if n_chunks == 1:
        work(0)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, range(n_chunks)))
    return out


def _scale_rows(rows: np.ndarray, scale: float, outlier, mult: float,
                chunk_rows: int = 65536, threads: int = 8) -> None:
    """In place on bf16 bits [n, width]: each row times `scale`, and rows where `outlier`
    is set times `mult` as well, rounded back to bf16 (nearest even).  Works block by
    block so that no full-size float32 copy is made; the values are those of the
    whole-array computation."""
    n = rows.shape[0]

    def work(lo):
        hi = min(n, lo + chunk_rows)
        f = bf16_bits_to_float32(rows[lo:hi]) * np.float32(scale)
        if outlier is not None:
            f[outlier[lo:hi]] *= np.float32(mult)
        rows[lo:hi] = _bf16_bits(f)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(work, range(0, n, chunk_rows)))


def random_tree(rng: np.random.Generator, T: int) -> np.ndarray:
    parent = np.full(T, -1, dtype=np.int64)
    for i in range(1, T):
        parent[i] = rng.integers(0, i)
    return parent


def chain_tree(T: int) -> np.ndarray:
    return np.arange(-1, T - 1, dtype=np.int64)


def tree_mask(parent: np.ndarray) -> np.ndarray:
    """[T, T] uint8: entry (i, j) = 1 iff j is i or an ancestor of i."""
    T = parent.shape[0]
    m = np.zeros((T, T), dtype=np.uint8)
    for i in range(T):
        j = i
        while j >= 0:
            m[i, j] = 1
            j = int(parent[j])
    return m


def build(name: str, seed: int, prefix_lens, draft_lens, tree: str, num_slots: int,
          heads: int = HEADS, q_scale: float = 1.0, kv_scale: float = 1.0,
          outlier_frac: float = 0.0, outlier_mult: float = 8.0,
          sm_scale: float = SM_SCALE, poison: bool = True,
          layout: str = "scattered") -> Workload:
    """Draws one workload.  ``tree`` is 'chain' or 'random'.

    ``layout`` places the referenced rows in the pool: 'scattered' (a random permutation
    of the slots, the default), 'contiguous' (all referenced rows in consecutive slots,
    request after request, as after a defragmenting gather-copy), or 'runs' (consecutive
    runs of 1 to 300 rows at random places).  Everything else is drawn identically."""
    prefix_lens = np.asarray(prefix_lens, dtype=np.int64)
    draft_lens = np.asarray(draft_lens, dtype=np.int64)
    bs = prefix_lens.shape[0]
    assert draft_lens.shape[0] == bs
    ss = np.random.SeedSequence(seed)
    s_meta, s_q, s_kv, s_out = ss.spawn(4)
    rng = np.random.default_rng(s_meta)

    L = prefix_lens + draft_lens
    n_ref = int(L.sum())
    if n_ref > num_slots:
        raise ValueError(f"{n_ref} referenced rows do not fit a {num_slots}-slot pool")
    slots = rng.permutation(num_slots)[:n_ref].astype(np.int64)
    if layout != "scattered":
        lay = np.random.default_rng([seed, 7])
        if layout == "contiguous":
            slots = int(lay.integers(0, num_slots - n_ref + 1)) + np.arange(n_ref, dtype=np.int64)
        elif layout == "runs":
            cuts = [0]
            while cuts[-1] < n_ref:
                cuts.append(min(n_ref, cuts[-1] + int(lay.integers(1, 301))))
            nruns = len(cuts) - 1
            # runs in random order over disjoint slot ranges: the pool is split into
            # nruns equal strides and each run starts at a random place in its own stride
            stride = num_slots // nruns
            order = lay.permutation(nruns)
            slots = np.empty(n_ref, dtype=np.int64)
            for i in range(nruns):
                n = cuts[i + 1] - cuts[i]
                if n > stride:
                    raise ValueError("pool too small for the 'runs' layout")
                base = int(order[i]) * stride + int(lay.integers(0, stride - n + 1))
                slots[cuts[i]:cuts[i + 1]] = base + np.arange(n)
        else:
            raise ValueError(layout)

    kv_indptr = np.zeros(bs + 1, dtype=np.int64)
    kv_indptr[1:] = np.cumsum(prefix_lens)
    qo_indptr = np.zeros(bs + 1, dtype=np.int64)
    qo_indptr[1:] = np.cumsum(draft_lens)
    if kv_indptr[-1] >= 2**31:
        raise ValueError("kv_indptr is int32")
    kv_indices = np.empty(int(kv_indptr[-1]), dtype=np.int32)
    out_cache_loc = np.empty(int(qo_indptr[-1]), dtype=np.int64)
    pos = 0
    for b in range(bs):
        P, T = int(prefix_lens[b]), int(draft_lens[b])
        kv_indices[kv_indptr[b]:kv_indptr[b + 1]] = slots[pos:pos + P]
        out_cache_loc[qo_indptr[b]:qo_indptr[b + 1]] = slots[pos + P:pos + P + T]
        pos += P + T

    parents = []
    mask_indptr = np.zeros(bs + 1, dtype=np.int64)
    blocks = []
    for b in range(bs):
        P, T = int(prefix_lens[b]), int(draft_lens[b])
        if tree == "chain":
            par = chain_tree(T)
        elif tree == "random":
            par = random_tree(rng, T)
        else:
            raise ValueError(tree)
        parents.append(par)
        blk = np.ones((T, P + T), dtype=np.uint8)
        blk[:, P:] = tree_mask(par)
        blocks.append(blk.reshape(-1))
        mask_indptr[b + 1] = mask_indptr[b] + T * (P + T)
    custom_mask = np.concatenate(blocks) if blocks else np.zeros(0, np.uint8)

    total_q = int(qo_indptr[-1])
    q = _normal_bf16(s_q, total_q * heads, D_QK)
    kv_rows = _normal_bf16(s_kv, n_ref, D_QK)
    if q_scale != 1.0 or kv_scale != 1.0 or outlier_frac > 0.0:
        ro = np.random.default_rng(s_out)
        kv_out = ro.random(n_ref) < outlier_frac if outlier_frac > 0.0 else None
        q_out = ro.random(total_q * heads) < outlier_frac if outlier_frac > 0.0 else None
        _scale_rows(kv_rows, kv_scale, kv_out, outlier_mult)
        _scale_rows(q, q_scale, q_out, outlier_mult)
    q = q.reshape(total_q, heads, D_QK)

    kv_cache = np.empty((num_slots, D_QK), dtype=np.uint16)
    kv_cache[...] = BF16_NAN if poison else np.uint16(0)
    kv_cache[slots] = kv_rows

    return Workload(name=name, q=q, kv_cache=kv_cache, kv_indices=kv_indices,
                    kv_indptr=kv_indptr.astype(np.int32), out_cache_loc=out_cache_loc,
                    custom_mask=custom_mask, mask_indptr=mask_indptr, qo_indptr=qo_indptr,
                    parents=parents, sm_scale=sm_scale)


def shape_sample(k: int, bs: int, heads: int = HEADS, layout: str = "scattered") -> Workload:
    """A smaller draw of shape k's distribution: `bs` requests instead of the shape's own
    batch, the pool scaled by the same factor (so the referenced rows fill the same share of
    it), another seed.  For profiling a small case of the same kind as a large shape."""
    seed = 20261300 + k
    rng = np.random.default_rng(seed + 1_000_000)
    if k == 4:
        P = np.exp(rng.uniform(math.log(512), math.log(32768), size=bs)).astype(np.int64)
        return build(f"bs{bs}_sample_of_shape4", seed, P, [8] * bs, "chain",
                     max(1 << 14, (1 << 20) * bs // 32), heads, layout=layout)
    if k == 5:
        P = rng.integers(8192, 65536, size=bs, endpoint=True)
        T = rng.choice(np.array([1, 4, 8, 16]), size=bs)
        return build(f"bs{bs}_sample_of_shape5", seed, P, T, "random",
                     max(1 << 16, (1 << 22) * bs // 64), heads, q_scale=0.5, kv_scale=0.5,
                     outlier_frac=0.01, outlier_mult=8.0, layout=layout)
    raise ValueError(f"no sampled form of shape {k}")


# The five shapes of the verify workload: (description, builder).  Seeds are
# 20261200 + the shape number.
def shape(k: int, heads: int = HEADS, layout: str = "scattered") -> Workload:
    seed = 20261200 + k
    rng = np.random.default_rng(seed + 1_000_000)  # sizes only
    if k == 1:
        return build("bs1_P128_T4_chain_pool4096", seed, [128], [4], "chain", 4096, heads,
                     layout=layout)
    if k == 2:
        P = rng.integers(1024, 4096, size=8, endpoint=True)
        return build("bs8_P1k-4k_T16_tree_pool65536", seed, P, [16] * 8, "random", 65536, heads,
                     layout=layout)
    if k == 3:
        return build("bs1_P185000_T16_tree_pool262144", seed, [185000], [16], "random", 262144, heads,
                     layout=layout)
    if k == 4:
        P = np.exp(rng.uniform(math.log(512), math.log(32768), size=32)).astype(np.int64)
        return build("bs32_P512-32k_logU_T8_chain_pool1M", seed, P, [8] * 32, "chain", 1 << 20, heads,
                     layout=layout)
    if k == 5:
        P = rng.integers(8192, 65536, size=64, endpoint=True)
        T = rng.choice(np.array([1, 4, 8, 16]), size=64)
        return build("bs64_P8k-64k_Tmix_tree_outliers_pool4M", seed, P, T, "random", 1 << 22, heads,
                     q_scale=0.5, kv_scale=0.5, outlier_frac=0.01, outlier_mult=8.0, layout=layout)
    raise ValueError(k)


SHAPE_NAMES = {
    1: "bs1_P128_T4_chain_pool4096",
    2: "bs8_P1k-4k_T16_tree_pool65536",
    3: "bs1_P185000_T16_tree_pool262144",
    4: "bs32_P512-32k_logU_T8_chain_pool1M",
    5: "bs64_P8k-64k_Tmix_tree_outliers_pool4M",
}
