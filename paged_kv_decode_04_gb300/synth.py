"""Seeded synthetic workloads for the paged-KV decode path.

This module only *draws* inputs: sequence lengths, random page assignments, and
N(0, 1) values rounded to bf16.  It holds none of the method's arithmetic (no
RoPE, no softmax, no attention), so both the CUDA path and the CPU oracle can
be fed from it without sharing any of the computation under test.

bf16 data is kept as raw ``uint16`` bit patterns on the host.  Unused pool
pages, and the slots of a live page at or beyond the appended position, hold
the poison pattern ``0xFFFF`` (a bf16 NaN) so that any read the method should
not make turns a result into NaN.

Workload shapes follow the Tiny-vLLM model dimensions (Llama 3.2 1B: 32 query
heads, 8 kv heads, head dim 64, 16-token pages, 2048-token context) from the
"Hours of YouTube and 85 handtyped pages of notes on LLM Inference - Start
here" README, sections "これまでの進捗" and "現在のスコープ".
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

POISON = 0xFFFF
NUM_Q_HEADS = 32
NUM_KV_HEADS = 8
HEAD_DIM = 64
PAGE_SIZE = 16
MAX_BLOCKS = 128  # 2048-token context / 16-token pages
ROPE_THETA = 500000.0
SCALE = 0.125  # 1 / sqrt(64)


@dataclass
class Workload:
    name: str
    seed: int
    layers: int
    batch: int
    num_pages: int
    seq_lens: np.ndarray          # int32 [B]; length after this step's append
    block_tables: np.ndarray      # int32 [layers][B][max_blocks]; -1 beyond the live blocks
    live_pages: np.ndarray        # int64 [n_live]; physical ids in (layer, seq, block) order
    page_data: np.ndarray         # uint16 [n_live][2][page_size][Hkv][D]; before the append
    q: np.ndarray                 # uint16 [layers][B][Hq][D]
    k_new: np.ndarray             # uint16 [layers][B][Hkv][D]
    v_new: np.ndarray             # uint16 [layers][B][Hkv][D]
    num_q_heads: int = NUM_Q_HEADS
    num_kv_heads: int = NUM_KV_HEADS
    head_dim: int = HEAD_DIM
    page_size: int = PAGE_SIZE
    max_blocks: int = MAX_BLOCKS
    rope_theta: float = ROPE_THETA
    scale: float = SCALE
    meta: dict = field(default_factory=dict)

    @property
    def positions(self) -> np.ndarray:
        """Decode position of the appended token: the last position of each sequence."""
        return (self.seq_lens.astype(np.int32) - 1).astype(np.int32)

    def pages_of(self, layer: int, b: int) -> np.ndarray:
        n = _num_blocks(int(self.seq_lens[b]), self.page_size)
        return self.block_tables[layer, b, :n]

    def kv_bytes(self) -> int:
        """Bytes of live K/V a full step streams: sum of lengths x Hkv x D x 2 (K,V) x 2 B."""
        return int(self.layers * int(self.seq_lens.astype(np.int64).sum())
                   * self.num_kv_heads * self.head_dim * 2 * 2)


def _num_blocks(L: int, page_size: int) -> int:
    return (max(L, 0) + page_size - 1) // page_size


def _bf16_normal(gen: torch.Generator, n: int) -> np.ndarray:
    """n draws of N(0, 1) in float32, rounded to bf16, as uint16 bits."""
    x = torch.randn(n, generator=gen, dtype=torch.float32)
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _lengths(name: str, rng: np.random.Generator, batch: int) -> np.ndarray:
    if name == "tiny":
        return np.full(batch, 37, dtype=np.int32)
    if name in ("long", "peak", "prefix"):
        return np.full(batch, 2048, dtype=np.int32)
    if name == "small":
        return rng.integers(1, 2048, size=batch, endpoint=True).astype(np.int32)
    if name == "mix":
        n_long = int(round(0.1 * batch))
        short = rng.integers(16, 128, size=batch - n_long, endpoint=True)
        long_ = rng.integers(1536, 2048, size=n_long, endpoint=True)
        lens = np.concatenate([short, long_]).astype(np.int32)
        rng.shuffle(lens)
        return lens
    raise ValueError(f"unknown workload {name!r}")


# name -> (layers, batch, pool pages) of each named workload.
WORKLOADS = {
    "tiny": (1, 1, 64),
    "long": (16, 1, 4096),
    "small": (1, 8, 4096),
    "peak": (1, 256, 40000),
    "mix": (16, 128, 262144),
    "prefix": (1, 256, 40000),
}
WORKLOAD_INDEX = {"tiny": 0, "long": 1, "small": 2, "peak": 3, "mix": 4, "prefix": 5}
# "prefix": consecutive groups of PREFIX_GROUP sequences share their first
# PREFIX_BLOCKS pages (a common 1536-token prompt prefix).
PREFIX_GROUP = 16
PREFIX_BLOCKS = 96


def make_workload(name: str, seed: int = 0, *, seq_lens=None, batch=None, layers=None,
                  num_pages=None, max_blocks: int = MAX_BLOCKS, share_group: int = None,
                  share_blocks: int = None) -> Workload:
    """Draw one of the named workloads (or a custom one via the keyword overrides).

    The seed mixes in the workload's index so that different workloads drawn
    with the same seed are independent.  With share_group = G and
    share_blocks = S, consecutive groups of G sequences alias the same S
    physical pages as their first S blocks (a shared prompt prefix); every
    sequence must then be longer than S pages' worth of tokens.
    """
    if name == "prefix" and share_group is None:
        share_group, share_blocks = PREFIX_GROUP, PREFIX_BLOCKS
    if name in WORKLOADS:
        d_layers, d_batch, d_pages = WORKLOADS[name]
        mix = WORKLOAD_INDEX[name]
    else:
        d_layers, d_batch, d_pages = 1, 1, 64
        mix = 97
    layers = d_layers if layers is None else layers
    num_pages = d_pages if num_pages is None else num_pages
    full_seed = int(seed) * 1000 + mix
    rng = np.random.default_rng(full_seed)
    if seq_lens is None:
        batch = d_batch if batch is None else batch
        seq_lens = _lengths(name, rng, batch)
    else:
        seq_lens = np.asarray(seq_lens, dtype=np.int32)
        batch = int(seq_lens.shape[0])
    if np.any(seq_lens > max_blocks * PAGE_SIZE):
        raise ValueError("sequence longer than the block table allows")
    blocks = [_num_blocks(int(L), PAGE_SIZE) for L in seq_lens]
    share_group = share_group or 1
    share_blocks = share_blocks or 0
    if share_blocks and any(int(L) <= share_blocks * PAGE_SIZE for L in seq_lens):
        raise ValueError("shared prefixes need every sequence longer than the shared pages")
    followers = batch - (-(-batch // share_group)) if share_blocks else 0
    n_live = layers * (sum(blocks) - followers * share_blocks)
    if n_live > num_pages:
        raise ValueError(f"{n_live} live pages do not fit a {num_pages}-page pool")

    gen = torch.Generator().manual_seed(full_seed)
    perm = torch.randperm(num_pages, generator=gen).numpy().astype(np.int64)
    live = perm[:n_live]

    bt = np.full((layers, batch, max_blocks), -1, dtype=np.int32)
    cursor = 0
    owned = []  # (b, first owned block, blocks) for each run of live pages, in order
    for layer in range(layers):
        for b in range(batch):
            n = blocks[b]
            first = 0
            if share_blocks and b % share_group != 0:
                lead = b - b % share_group  # alias the group leader's prefix pages
                bt[layer, b, :share_blocks] = bt[layer, lead, :share_blocks]
                first = share_blocks
            bt[layer, b, first:n] = live[cursor:cursor + n - first]
            owned.append((b, first, n))
            cursor += n - first

    Hq, Hkv, D, P = NUM_Q_HEADS, NUM_KV_HEADS, HEAD_DIM, PAGE_SIZE
    page_elems = 2 * P * Hkv * D
    page_data = np.empty((n_live, 2, P, Hkv, D), dtype=np.uint16)
    flat = page_data.reshape(n_live, page_elems)
    chunk = 2048
    for s in range(0, n_live, chunk):
        e = min(n_live, s + chunk)
        flat[s:e] = _bf16_normal(gen, (e - s) * page_elems).reshape(e - s, page_elems)
    # Poison every slot at or past the appended position (position L-1) of each
    # sequence's last page; the append step writes position L-1 itself.
    cursor = 0
    for b, first, n in owned:
        if n > first:
            first_dead = (int(seq_lens[b]) - 1) % P
            page_data[cursor + n - first - 1, :, first_dead:, :, :] = POISON
        cursor += n - first

    q = _bf16_normal(gen, layers * batch * Hq * D).reshape(layers, batch, Hq, D)
    k_new = _bf16_normal(gen, layers * batch * Hkv * D).reshape(layers, batch, Hkv, D)
    v_new = _bf16_normal(gen, layers * batch * Hkv * D).reshape(layers, batch, Hkv, D)
    return Workload(name=name, seed=int(seed), layers=layers, batch=batch, num_pages=num_pages,
                    seq_lens=seq_lens, block_tables=bt, live_pages=live, page_data=page_data,
                    q=q, k_new=k_new, v_new=v_new, max_blocks=max_blocks,
                    meta={"full_seed": full_seed})


# ------------------------------------------------------------ host views --

def host_pool(w: Workload) -> np.ndarray:
    """The whole physical pool on the host (small pools only): poison + live pages."""
    pool = np.full((w.num_pages, 2, w.page_size, w.num_kv_heads, w.head_dim), POISON,
                   dtype=np.uint16)
    pool[w.live_pages] = w.page_data
    return pool


@dataclass
class Compact:
    """A relabelled copy of some sequences of one layer for the oracle.

    ``pool`` holds only the pages those sequences use, and ``block_table`` maps
    their blocks to indices in that compact pool (a pure relabelling of pages).
    """
    seqs: np.ndarray
    pool: np.ndarray
    block_table: np.ndarray
    seq_lens: np.ndarray
    positions: np.ndarray
    q: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray


def compact(w: Workload, layer: int, seqs=None) -> Compact:
    seqs = np.arange(w.batch) if seqs is None else np.asarray(seqs, dtype=np.int64)
    # index of each physical page in page_data (-1: not live)
    index_of = np.full(w.num_pages, -1, dtype=np.int64)
    index_of[w.live_pages] = np.arange(len(w.live_pages), dtype=np.int64)
    bt = np.full((len(seqs), w.max_blocks), -1, dtype=np.int32)
    chunks = []
    count = 0
    for r, b in enumerate(seqs):
        ids = w.pages_of(layer, int(b)).astype(np.int64)
        bt[r, :len(ids)] = np.arange(count, count + len(ids), dtype=np.int32)
        chunks.append(index_of[ids])
        count += len(ids)
    pages = np.concatenate(chunks) if count else np.zeros(0, dtype=np.int64)
    if np.any(pages < 0):
        raise ValueError("a block table names a page that holds no live data")
    pool = w.page_data[pages] if count else np.zeros(
        (0, 2, w.page_size, w.num_kv_heads, w.head_dim), dtype=np.uint16)
    pool = np.ascontiguousarray(pool)
    return Compact(seqs=seqs, pool=pool, block_table=bt,
                   seq_lens=w.seq_lens[seqs].copy(), positions=w.positions[seqs].copy(),
                   q=np.ascontiguousarray(w.q[layer][seqs]),
                   k_new=np.ascontiguousarray(w.k_new[layer][seqs]),
                   v_new=np.ascontiguousarray(w.v_new[layer][seqs]))


# --------------------------------------------------------------- prefill --

@dataclass
class Prefill:
    """A ragged prefill batch: prompt b's tokens [token_offsets[b],
    token_offsets[b+1]) of k and v go to positions start_positions[b] + i
    through block_table row b (the prompt's pages, randomly scattered)."""
    batch: int
    prompt_len: int
    num_pages: int
    k: np.ndarray                 # uint16 [tokens][Hkv][D]
    v: np.ndarray                 # uint16 [tokens][Hkv][D]
    token_offsets: np.ndarray     # int32 [B + 1]
    start_positions: np.ndarray   # int32 [B]
    block_table: np.ndarray       # int32 [B][max_blocks]


def make_prefill(seed: int = 0, batch: int = 256, prompt_len: int = 2047,
                 num_pages: int = 40000, max_blocks: int = MAX_BLOCKS) -> Prefill:
    """batch prompts of prompt_len tokens each, written from position 0; every
    prompt owns ceil(prompt_len / 16) pages of a random permutation of the pool."""
    full_seed = int(seed) * 1000 + 96
    gen = torch.Generator().manual_seed(full_seed)
    blocks = _num_blocks(prompt_len, PAGE_SIZE)
    if batch * blocks > num_pages or blocks > max_blocks:
        raise ValueError("the prompts do not fit the pool or the block table")
    perm = torch.randperm(num_pages, generator=gen).numpy().astype(np.int32)
    bt = np.full((batch, max_blocks), -1, dtype=np.int32)
    bt[:, :blocks] = perm[:batch * blocks].reshape(batch, blocks)
    n = batch * prompt_len * NUM_KV_HEADS * HEAD_DIM
    k = _bf16_normal(gen, n).reshape(batch * prompt_len, NUM_KV_HEADS, HEAD_DIM)
    v = _bf16_normal(gen, n).reshape(batch * prompt_len, NUM_KV_HEADS, HEAD_DIM)
    offsets = np.arange(0, batch * prompt_len + 1, prompt_len, dtype=np.int32)
    return Prefill(batch=batch, prompt_len=prompt_len, num_pages=num_pages, k=k, v=v,
                   token_offsets=offsets, start_positions=np.zeros(batch, dtype=np.int32),
                   block_table=bt)


@dataclass
class CompactPrefill:
    """Some prompts of a Prefill relabelled onto a pool of only their pages
    (poison-filled), for the oracle: pages[i] is the physical page of compact
    page i."""
    pages: np.ndarray
    pool: np.ndarray
    k: np.ndarray
    v: np.ndarray
    token_offsets: np.ndarray
    start_positions: np.ndarray
    block_table: np.ndarray


def compact_prefill(p: Prefill, prompts) -> CompactPrefill:
    prompts = [int(b) for b in prompts]
    blocks = _num_blocks(p.prompt_len, PAGE_SIZE)
    bt = np.full((len(prompts), p.block_table.shape[1]), -1, dtype=np.int32)
    bt[:, :blocks] = np.arange(len(prompts) * blocks, dtype=np.int32).reshape(-1, blocks)
    pages = np.concatenate([p.block_table[b, :blocks] for b in prompts]).astype(np.int64)
    ks = np.concatenate([p.k[p.token_offsets[b]:p.token_offsets[b + 1]] for b in prompts])
    vs = np.concatenate([p.v[p.token_offsets[b]:p.token_offsets[b + 1]] for b in prompts])
    lens = [int(p.token_offsets[b + 1] - p.token_offsets[b]) for b in prompts]
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    pool = np.full((len(pages), 2, PAGE_SIZE, NUM_KV_HEADS, HEAD_DIM), POISON, dtype=np.uint16)
    return CompactPrefill(pages=pages, pool=pool, k=np.ascontiguousarray(ks),
                          v=np.ascontiguousarray(vs), token_offsets=offsets,
                          start_positions=p.start_positions[prompts].copy(), block_table=bt)


# ---------------------------------------------------------- device views --

def to_device_bf16(a: np.ndarray, device) -> torch.Tensor:
    """uint16 bf16 bit patterns -> a bf16 tensor on `device`."""
    return _to_bf16_tensor(a, device)



def _to_bf16_tensor(a: np.ndarray, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def device_inputs(w: Workload, device="cuda") -> dict:
    """Upload a workload: the poison-filled pool with live pages scattered in,
    per-layer tables, queries, new K/V, lengths and positions."""
    Hkv, D, P = w.num_kv_heads, w.head_dim, w.page_size
    pool = torch.full((w.num_pages, 2, P, Hkv, D), -1, dtype=torch.int16, device=device)
    live = torch.from_numpy(w.live_pages).to(device)
    chunk = 4096
    for s in range(0, len(w.live_pages), chunk):
        e = min(len(w.live_pages), s + chunk)
        pool[live[s:e]] = torch.from_numpy(w.page_data[s:e].view(np.int16)).to(device)
    return {
        "pool": pool.view(torch.bfloat16),
        "block_tables": torch.from_numpy(w.block_tables).to(device),
        "q": _to_bf16_tensor(w.q, device),
        "k_new": _to_bf16_tensor(w.k_new, device),
        "v_new": _to_bf16_tensor(w.v_new, device),
        "seq_lens": torch.from_numpy(w.seq_lens.astype(np.int32)).to(device),
        "positions": torch.from_numpy(w.positions.astype(np.int32)).to(device),
    }


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor (copied to the host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
