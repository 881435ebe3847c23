"""Seeded synthetic workloads shaped like the pages' examples and workloads.

The pages name no public benchmark or dataset; every tensor here is drawn
from a CPU ``torch.Generator`` seeded per case (seed 1000 + workload number
for the five named workloads), so the CUDA path and the oracle read the same
bits.  Lengths, block placement and shared prefixes follow the structure the
pages describe:

* block tables map logical block i of a sequence to a physical block that
  may sit anywhere in the pool ("Perhatian berhalaman", Jalur decode /
  Contoh: blocks 3, 5, 6 are not adjacent), -1 beyond the allocated blocks;
* a sequence of cached length L needs ceil((L + 1) / block_size) blocks
  once the new token is appended (same example: 32 + 1 > 32 needs a second
  block);
* shared prefixes reuse the same physical blocks in many tables (the
  refcounted sharing of "Paged Attention", 共享前缀, and "PagedAttention",
  paweldubiel.com);
* varlen requests are packed along the token axis with exclusive cumulative
  lengths cu_seq_lens ("Perhatian berhalaman", Jalur Varlen / Contoh).

Nothing in this module computes attention.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

CONFIG_NAMES = {
    1: "tiny paged decode fp32: B=3 Hq=4 Hkv=2 D=64 bs=32 L=[30,32,70] table of the worked example",
    2: "paged decode bf16: B=64 Hq=32 Hkv=8 D=128 bs=16 L~U[512,4096]",
    3: "long-context paged decode bf16 (split-K): B=256 Hq=64 Hkv=8 D=128 bs=16 L~lognormal(median 2048) clipped [64,32768]",
    4: "varlen causal prefill + paged scatter bf16: 32 reqs ql~U[1,2048] prefix~U[0,1024] Hq=32 Hkv=8 D=128 bs=16",
    5: "shared-prefix mixed decode bf16: 1024 x (256 shared + U[1,512] private) + 4 x 131072, Hq=Hkv=32 D=64 bs=32",
}


def to_numpy(t: torch.Tensor) -> np.ndarray:
    """CPU tensor -> numpy; bfloat16 becomes its uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _randn(gen, shape, dtype, scale=1.0):
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(dtype)


@dataclass
class DecodeCase:
    q: torch.Tensor            # [B, Hq, D]
    k_cache: torch.Tensor      # [NB, bs, Hkv, D]
    v_cache: torch.Tensor
    block_table: torch.Tensor  # [B, MB] int32, -1 padded
    cache_seqlens: torch.Tensor  # [B] int32
    k_new: torch.Tensor        # [B, Hkv, D]
    v_new: torch.Tensor
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def batch(self):
        return self.q.shape[0]

    @property
    def num_heads(self):
        return self.q.shape[1]

    @property
    def head_dim(self):
        return self.q.shape[2]

    @property
    def num_blocks(self):
        return self.k_cache.shape[0]

    @property
    def block_size(self):
        return self.k_cache.shape[1]

    @property
    def num_kv_heads(self):
        return self.k_cache.shape[2]

    @property
    def max_blocks_per_seq(self):
        return self.block_table.shape[1]

    def elt(self):
        return self.q.element_size()

    def logical_kv_bytes(self) -> int:
        """K+V bytes the attention reads if every sequence counts its own."""
        t = self.cache_seqlens.to(torch.int64) + 1
        return int(t.sum()) * self.num_kv_heads * self.head_dim * self.elt() * 2

    def unique_kv_bytes(self) -> int:
        """K+V bytes of distinct pool rows read (a shared block counts once)."""
        bs = self.block_size
        tab = self.block_table.numpy()
        rows = []
        for b, L in enumerate(self.cache_seqlens.tolist()):
            pos = np.arange(L + 1)
            rows.append(tab[b, pos // bs].astype(np.int64) * bs + pos % bs)
        n = np.unique(np.concatenate(rows)).size
        return n * self.num_kv_heads * self.head_dim * self.elt() * 2

    def io_bytes(self) -> int:
        """q, out, k_new, v_new (read) and the appended rows (written)."""
        e = self.elt()
        b = self.batch
        return (2 * b * self.num_heads * self.head_dim + 4 * b * self.num_kv_heads *
                self.head_dim) * e

    def poison_unowned(self, value: float = float("nan")) -> "DecodeCase":
        """Fill every pool slot that holds none of the cached positions
        0..L_b-1 of any sequence with `value` (NaN by default): unused
        blocks, the tails of last blocks and the append slots, i.e. what a
        serving pool allocated with uninitialised memory may hold there.  The
        attended values are unchanged (the append slot is written before it
        is read).  In place; returns self."""
        bs = self.block_size
        tab = self.block_table.numpy()
        owned = np.zeros(self.num_blocks * bs, dtype=bool)
        for b, L in enumerate(self.cache_seqlens.tolist()):
            pos = np.arange(L)
            owned[tab[b, pos // bs].astype(np.int64) * bs + pos % bs] = True
        free = torch.from_numpy(~owned).view(self.num_blocks, bs)
        self.k_cache[free] = value
        self.v_cache[free] = value
        return self

    def contiguous_cache(self, max_seqlen=None, fill: float = float("nan"), device="cpu"):
        """The same logical K and V as a contiguous cache [B, max_seqlen,
        Hkv, D] (the input of the contiguous-cache decode twin): row b holds
        sequence b's cached positions 0..L_b-1, copied from the pool blocks
        its table names, and `fill` everywhere else.  Returns (k, v) on
        `device`."""
        bs = self.block_size
        L = self.cache_seqlens.to(torch.int64)
        lmax = int(max_seqlen or int(L.max()) + 1)
        pos = torch.arange(lmax)
        tab = self.block_table.to(torch.int64)
        blk = tab.gather(1, (pos // bs).clamp(max=tab.shape[1] - 1).expand(self.batch, -1))
        valid = pos.unsqueeze(0) < L.unsqueeze(1)
        rows = torch.where(valid, blk * bs + pos % bs, torch.zeros_like(blk)).reshape(-1)
        out = []
        for pool in (self.k_cache, self.v_cache):
            flat = pool.reshape(-1, self.num_kv_heads, self.head_dim).to(device)
            c = flat[rows.to(device)].reshape(self.batch, lmax, self.num_kv_heads, self.head_dim)
            c[~valid.to(device)] = fill
            out.append(c.contiguous())
        return out[0], out[1]

    def permuted(self, seed: int) -> "DecodeCase":
        """Same logical content with the physical blocks renumbered by a
        random permutation pi: block p moves to pi[p]."""
        g = torch.Generator().manual_seed(seed)
        pi = torch.randperm(self.num_blocks, generator=g)
        inv = torch.empty_like(pi)
        inv[pi] = torch.arange(self.num_blocks)
        k = self.k_cache[inv].clone()
        v = self.v_cache[inv].clone()
        tab = self.block_table.clone()
        m = tab >= 0
        tab[m] = pi[tab[m].long()].to(torch.int32)
        c = DecodeCase(self.q, k, v, tab, self.cache_seqlens, self.k_new, self.v_new,
                       self.name + f" (permuted {seed})", dict(self.meta, perm=pi))
        return c


def _place_blocks(gen, need, num_blocks, shared=None, contiguous=False):
    """Assign physical blocks: a seeded random permutation of the pool,
    handed out in order (or, with `contiguous`, the pool in order, so each
    sequence's blocks are adjacent, as a non-paged cache would lay them out).
    `shared` (list of physical ids) are reserved and given to rows flagged in
    need as (shared_count, private_count)."""
    perm = torch.randperm(num_blocks, generator=gen).tolist()
    if contiguous:
        perm = list(range(num_blocks))
    if shared:
        reserved = set(shared)
        perm = [p for p in perm if p not in reserved]
    tables = []
    off = 0
    for n_shared, n_priv in need:
        row = list(shared[:n_shared]) if n_shared else []
        row += perm[off:off + n_priv]
        off += n_priv
        tables.append(row)
    assert off <= len(perm), "pool too small"
    return tables


def _table_tensor(rows, mb):
    t = torch.full((len(rows), mb), -1, dtype=torch.int32)
    for i, r in enumerate(rows):
        t[i, :len(r)] = torch.tensor(r, dtype=torch.int32)
    return t


def make_decode(seed: int, lengths, num_heads: int, num_kv_heads: int, head_dim: int,
                block_size: int, dtype=torch.bfloat16, value_scale: float = 1.0,
                slack: float = 0.1, shared_prefix_blocks: int = 0, shared_rows=None,
                max_blocks_per_seq: int | None = None, block_table=None, num_blocks=None,
                name: str = "", contiguous: bool = False) -> DecodeCase:
    """Decode case with cached lengths `lengths` (keys before the append).

    Without an explicit `block_table`, row b gets ceil((L_b + 1) / bs)
    blocks; rows in `shared_rows` start with the same `shared_prefix_blocks`
    physical blocks.  The pool has (1 + slack) x the distinct blocks needed.
    """
    gen = torch.Generator().manual_seed(seed)
    lengths = [int(x) for x in lengths]
    b = len(lengths)
    if block_table is None:
        shared_rows = set(shared_rows or [])
        need = []
        for i, L in enumerate(lengths):
            n = -(-(L + 1) // block_size)
            ns = min(shared_prefix_blocks, n) if i in shared_rows else 0
            need.append((ns, n - ns))
        distinct = sum(p for _, p in need) + (shared_prefix_blocks if shared_rows else 0)
        nb = num_blocks or max(1, math.ceil((1.0 + slack) * distinct))
        shared = None
        if shared_rows and shared_prefix_blocks:
            shared = torch.randperm(nb, generator=gen)[:shared_prefix_blocks].tolist()
        rows = _place_blocks(gen, need, nb, shared, contiguous)
        mb = max_blocks_per_seq or max(len(r) for r in rows)
        table = _table_tensor(rows, mb)
    else:
        table = torch.as_tensor(block_table, dtype=torch.int32).clone()
        mb = table.shape[1]
        nb = int(num_blocks)
    q = _randn(gen, (b, num_heads, head_dim), dtype, value_scale)
    k_cache = _randn(gen, (nb, block_size, num_kv_heads, head_dim), dtype, value_scale)
    v_cache = _randn(gen, (nb, block_size, num_kv_heads, head_dim), dtype, value_scale)
    k_new = _randn(gen, (b, num_kv_heads, head_dim), dtype, value_scale)
    v_new = _randn(gen, (b, num_kv_heads, head_dim), dtype, value_scale)
    sl = torch.tensor(lengths, dtype=torch.int32)
    return DecodeCase(q, k_cache, v_cache, table, sl, k_new, v_new, name,
                      dict(seed=seed, value_scale=value_scale))


@dataclass
class VarlenCase:
    q: torch.Tensor            # [Tq, Hq, D]
    k_chunk: torch.Tensor      # [Tq, Hkv, D] new keys of every request
    v_chunk: torch.Tensor
    k_cache: torch.Tensor      # [NB, bs, Hkv, D] pool holding the cached prefixes
    v_cache: torch.Tensor
    block_table: torch.Tensor  # [B, MB]
    prefix_lens: torch.Tensor  # [B] int32
    cu_seq_lens_q: torch.Tensor  # [B+1] int32
    cu_seq_lens_k: torch.Tensor  # [B+1] int32 (prefix + chunk)
    max_length_q: int
    max_length_k: int
    causal: bool = True
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def batch(self):
        return len(self.prefix_lens)

    def poison_unowned(self, value: float = float("nan")) -> "VarlenCase":
        """Fill every pool slot that holds no cached prefix position of any
        request with `value` (NaN by default): the slots the chunk will be
        scattered into, the tails of last blocks and unused blocks.  In
        place; returns self."""
        bs = self.k_cache.shape[1]
        nb = self.k_cache.shape[0]
        tab = self.block_table.numpy()
        owned = np.zeros(nb * bs, dtype=bool)
        for r, L in enumerate(self.prefix_lens.tolist()):
            pos = np.arange(L)
            owned[tab[r, pos // bs].astype(np.int64) * bs + pos % bs] = True
        free = torch.from_numpy(~owned).view(nb, bs)
        self.k_cache[free] = value
        self.v_cache[free] = value
        return self

    def causal_pairs(self) -> int:
        """(query, key) pairs the bottom-right causal mask keeps."""
        cq = self.cu_seq_lens_q.tolist()
        ck = self.cu_seq_lens_k.tolist()
        tot = 0
        for r in range(self.batch):
            ql, kl = cq[r + 1] - cq[r], ck[r + 1] - ck[r]
            if not self.causal:
                tot += ql * kl
                continue
            i = np.arange(ql)
            tot += int(np.clip(i + kl - ql + 1, 0, kl).sum())
        return tot


def make_varlen(seed: int, q_lens, prefix_lens, num_heads: int, num_kv_heads: int,
                head_dim: int, block_size: int, dtype=torch.bfloat16, causal: bool = True,
                value_scale: float = 1.0, slack: float = 0.1, name: str = "") -> VarlenCase:
    """Requests with new-token counts `q_lens` after cached prefixes
    `prefix_lens`; each request owns ceil((prefix + q) / bs) pool blocks."""
    gen = torch.Generator().manual_seed(seed)
    q_lens = [int(x) for x in q_lens]
    prefix_lens = [int(x) for x in prefix_lens]
    k_lens = [a + b for a, b in zip(q_lens, prefix_lens)]
    need = [(0, -(-kl // block_size)) for kl in k_lens]
    nb = max(1, math.ceil((1.0 + slack) * sum(n for _, n in need)))
    rows = _place_blocks(gen, need, nb)
    mb = max(1, max(len(r) for r in rows))
    table = _table_tensor(rows, mb)
    tq = sum(q_lens)
    q = _randn(gen, (tq, num_heads, head_dim), dtype, value_scale)
    k_chunk = _randn(gen, (tq, num_kv_heads, head_dim), dtype, value_scale)
    v_chunk = _randn(gen, (tq, num_kv_heads, head_dim), dtype, value_scale)
    k_cache = _randn(gen, (nb, block_size, num_kv_heads, head_dim), dtype, value_scale)
    v_cache = _randn(gen, (nb, block_size, num_kv_heads, head_dim), dtype, value_scale)
    cu_q = torch.tensor([0] + list(np.cumsum(q_lens)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(np.cumsum(k_lens)), dtype=torch.int32)
    return VarlenCase(q, k_chunk, v_chunk, k_cache, v_cache, table,
                      torch.tensor(prefix_lens, dtype=torch.int32), cu_q, cu_k,
                      max(q_lens) if q_lens else 0, max(k_lens) if k_lens else 0, causal, name,
                      dict(seed=seed))


# --------------------------------------------------------------------------
# the five named workloads
# --------------------------------------------------------------------------

WORKED_EXAMPLE_TABLE = [[2, -1, -1, -1], [0, 1, -1, -1], [3, 5, 6, -1]]
WORKED_EXAMPLE_SEQLENS = [30, 32, 70]


def decode_config(idx: int, scale_down: int = 1, seed_offset: int = 0,
                  contiguous: bool = False, unit_variance: bool = False) -> DecodeCase:
    """Decode workloads 1, 2, 3 and 5.  `scale_down` > 1 keeps the structure
    (heads, head_dim, block size, length distribution) with fewer sequences,
    for oracle runs that must finish in seconds.  `seed_offset` draws another
    batch of the same workload (one per rank when the benchmark runs on
    several GPUs).  `unit_variance` draws workload 2's values N(0,1) instead
    of N(0,1)/sqrt(128): the same shapes with outputs large enough that a
    wrong result cannot hide under the absolute tolerance."""
    seed = 1000 + idx + 100 * seed_offset
    if idx == 1:
        return make_decode(seed, WORKED_EXAMPLE_SEQLENS, 4, 2, 64, 32, dtype=torch.float32,
                           block_table=WORKED_EXAMPLE_TABLE, num_blocks=8, name=CONFIG_NAMES[1])
    g = torch.Generator().manual_seed(seed + 50_000)
    if idx == 2:
        b = max(1, 64 // scale_down)
        lengths = torch.randint(512, 4097, (b,), generator=g).tolist()
        vs = 1.0 if unit_variance else 1.0 / math.sqrt(128.0)
        name = CONFIG_NAMES[2] + (" (blocks contiguous)" if contiguous else "") + (
            " (values N(0,1))" if unit_variance else "")
        return make_decode(seed, lengths, 32, 8, 128, 16, value_scale=vs, name=name,
                           contiguous=contiguous)
    if idx == 3:
        b = max(1, 256 // scale_down)
        z = torch.randn(b, generator=g, dtype=torch.float64)
        lengths = torch.exp(math.log(2048.0) + 1.0 * z).round().clamp(64, 32768)
        return make_decode(seed, lengths.to(torch.int64).tolist(), 64, 8, 128, 16,
                           name=CONFIG_NAMES[3] + (" (blocks contiguous)" if contiguous else ""),
                           contiguous=contiguous)
    if idx == 5:
        n_short = max(1, 1024 // scale_down)
        n_long = 4 if scale_down == 1 else 1
        long_len = 131072 if scale_down == 1 else max(2048, 131072 // scale_down)
        priv = torch.randint(1, 513, (n_short,), generator=g).tolist()
        lengths = [256 + p for p in priv] + [long_len] * n_long
        return make_decode(seed, lengths, 32, 32, 64, 32, shared_prefix_blocks=8,
                           shared_rows=range(n_short), name=CONFIG_NAMES[5])
    raise ValueError(f"no decode workload {idx}")


def varlen_config(idx: int = 4, scale_down: int = 1) -> VarlenCase:
    if idx != 4:
        raise ValueError("workload 4 is the varlen one")
    seed = 1000 + idx
    g = torch.Generator().manual_seed(seed + 50_000)
    b = max(1, 32 // scale_down)
    qmax = max(2, 2048 // scale_down)
    pmax = 1024 // scale_down
    q_lens = torch.randint(1, qmax + 1, (b,), generator=g).tolist()
    prefix = torch.randint(0, pmax + 1, (b,), generator=g).tolist()
    return make_varlen(seed, q_lens, prefix, 32, 8, 128, 16, name=CONFIG_NAMES[4])
