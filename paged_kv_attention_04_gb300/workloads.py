"""Seeded synthetic inputs for one continuous-batching attention step.

This module builds the inputs only: request lengths, block tables, the slot
mapping, the new tokens' Q/K/V and a paged KV pool whose history slots hold
N(0, 1) data.  It holds none of the attention arithmetic, so both the fp64
oracle and the CUDA path can take their inputs from here.

Structure follows the pages:
  * a KV block holds 16 tokens; a request with n tokens owns ceil(n/16)
    blocks ("Inside vLLM", section Scheduler, allocate_slots);
  * a request's block table lists its physical blocks in logical order and
    they need not be contiguous ("Serving models at scale with vLLM",
    section PagedAttention: Req 2 -> blocks 2, 5, 8);
  * a token's slot is its physical block * 16 + its offset in that block,
    built on the host in "prepare inputs" ("Inside vLLM", section Run
    forward pass);
  * the step is one flattened super-sequence, decodes first, then chunked
    prefills ("Serving models at scale with vLLM", section Chunked prefill);
  * full blocks of a shared prefix may be mapped by several block tables
    ("LLM Serving Frameworks #1", section 4, KVCacheManager: #42 shared).

Host metadata comes from numpy's PCG64 (platform independent); tensor data
comes from a torch.Generator on the chosen device.  Every slot that holds no
history (unused pool blocks, the slots this step writes, slots past a
request's length) is NaN, so a stray read poisons the result.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK_SIZE = 16


@dataclass
class StepSpec:
    """Shape of one step: heads, head size, dtype and per-request lengths."""
    name: str
    dtype: str                      # "f32" or "bf16"
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    q_lens: np.ndarray              # int64 [B], new tokens per request
    seq_lens: np.ndarray            # int64 [B], KV length incl. the new tokens
    num_blocks: int | None = None   # pool size; None -> ceil(pool_factor * needed)
    pool_factor: float = 1.2
    shared_prefix_blocks: int = 0   # physical blocks shared by `sharing` requests
    sharing: np.ndarray | None = None  # bool [B]
    seed: int = 0
    block_size: int = BLOCK_SIZE

    @property
    def num_seqs(self) -> int:
        return int(len(self.seq_lens))

    @property
    def num_tokens(self) -> int:
        return int(self.q_lens.sum())


@dataclass
class Step:
    """All inputs of one step.  Tensors live on `device`."""
    spec: StepSpec
    num_blocks: int
    block_tables: torch.Tensor      # int32 [B][max_blocks], -1 past the end
    seq_lens: torch.Tensor          # int32 [B]
    query_start_loc: torch.Tensor   # int32 [B+1]
    slot_mapping: torch.Tensor      # int64 [T]
    q: torch.Tensor                 # [T][Hq][D]
    k: torch.Tensor                 # [T][Hkv][D]  new keys
    v: torch.Tensor                 # [T][Hkv][D]  new values
    k_cache: torch.Tensor           # [NB][16][Hkv][D]
    v_cache: torch.Tensor           # [NB][16][Hkv][D]
    scale: float
    unique_blocks: int = 0          # physical blocks referenced by some table
    meta: dict = field(default_factory=dict)

    @property
    def max_seq_len(self) -> int:
        return int(self.spec.seq_lens.max()) if self.spec.num_seqs else 0

    @property
    def max_query_len(self) -> int:
        return int(self.spec.q_lens.max()) if self.spec.num_seqs else 0

    def to(self, device) -> "Step":
        out = Step(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        for name in ("block_tables", "seq_lens", "query_start_loc", "slot_mapping",
                     "q", "k", "v", "k_cache", "v_cache"):
            setattr(out, name, getattr(self, name).to(device))
        return out


# --------------------------------------------------------------------------
# The five workloads.  Lengths use inclusive integer ranges; "context" is the
# KV length a request attends to in this step, the new token included.
# --------------------------------------------------------------------------

def spec_tiny_decode_f32(seed: int = 0) -> StepSpec:
    """4 decode requests, seq_lens {1,17,33,64}, 4 q / 2 kv heads, D=64, fp32,
    a 32-block pool with non-contiguous tables."""
    seq = np.array([1, 17, 33, 64], dtype=np.int64)
    return StepSpec("tiny_decode_f32", "f32", 4, 2, 64, np.ones(4, np.int64), seq,
                    num_blocks=32, seed=seed)


def spec_tinyllama_decode(seed: int = 1) -> StepSpec:
    """TinyLlama-1.1B layer shape: batch 64, 32 q / 4 kv heads, D=64, bf16,
    context uniform in [128, 2048], pool 1.2x the blocks needed."""
    rng = np.random.default_rng(seed)
    seq = rng.integers(128, 2048, size=64, endpoint=True).astype(np.int64)
    return StepSpec("tinyllama_decode", "bf16", 32, 4, 64, np.ones(64, np.int64), seq,
                    seed=seed)


def spec_llama3_8b_decode(seed: int = 2) -> StepSpec:
    """Llama-3-8B layer shape: batch 256, 32 q / 8 kv heads, D=128, bf16,
    context lognormal (median 1024, sigma 0.8) capped at 8192."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal(256)
    seq = np.clip(np.rint(np.exp(math.log(1024.0) + 0.8 * z)), 1, 8192).astype(np.int64)
    return StepSpec("llama3_8b_decode", "bf16", 32, 8, 128, np.ones(256, np.int64), seq,
                    seed=seed)


def spec_mixed_step(seed: int = 3) -> StepSpec:
    """Mixed step, Llama-3-8B heads, bf16: 192 decodes (context uniform in
    [256, 4096]) then two 512-token prefill chunks with prior context 0 and
    1536; token budget 1216.  A seeded half of the decodes map their first
    min(64, (S-1)//16) logical blocks onto one shared set of 64 blocks."""
    rng = np.random.default_rng(seed)
    dec = rng.integers(256, 4096, size=192, endpoint=True).astype(np.int64)
    seq = np.concatenate([dec, np.array([512, 1536 + 512], np.int64)])
    ql = np.concatenate([np.ones(192, np.int64), np.array([512, 512], np.int64)])
    sharing = np.zeros(194, dtype=bool)
    sharing[rng.choice(192, size=96, replace=False)] = True
    return StepSpec("mixed_step", "bf16", 32, 8, 128, ql, seq,
                    shared_prefix_blocks=64, sharing=sharing, seed=seed)


def spec_long_context_decode(seed: int = 4) -> StepSpec:
    """Long-context decode: batch 16, context uniform in [32768, 131072],
    32 q / 8 kv heads, D=128, bf16, a pool of floor(9e9 / 65536) blocks."""
    rng = np.random.default_rng(seed)
    seq = rng.integers(32768, 131072, size=16, endpoint=True).astype(np.int64)
    return StepSpec("long_context_decode", "bf16", 32, 8, 128, np.ones(16, np.int64), seq,
                    num_blocks=int(9e9 // 65536), seed=seed)


def spec_long_prefill_chunk(seed: int = 5) -> StepSpec:
    """One 2048-token prefill chunk of a long prompt: prior context 6144, so
    the chunk's rows see up to 8192 keys; Llama-3-8B heads, bf16."""
    return StepSpec("long_prefill_chunk", "bf16", 32, 8, 128, np.array([2048], np.int64),
                    np.array([8192], np.int64), seed=seed)


def spec_long_prior_chunks(seed: int = 6) -> StepSpec:
    """Short prefill chunks late in long prompts: a 64-token chunk after 32768
    tokens and a 16-token chunk after 98304 ("Serving models at scale with
    vLLM", section Chunked prefill: a long prompt is split under a small token
    budget and every later chunk reads all earlier ones from the cache);
    Llama-3-8B heads, bf16."""
    return StepSpec("long_prior_chunks", "bf16", 32, 8, 128, np.array([64, 16], np.int64),
                    np.array([32768 + 64, 98304 + 16], np.int64), seed=seed)


CONFIGS = {
    "tiny_decode_f32": spec_tiny_decode_f32,
    "tinyllama_decode": spec_tinyllama_decode,
    "llama3_8b_decode": spec_llama3_8b_decode,
    "mixed_step": spec_mixed_step,
    "long_context_decode": spec_long_context_decode,
    "long_prefill_chunk": spec_long_prefill_chunk,
    "long_prior_chunks": spec_long_prior_chunks,
}


def custom_spec(name: str, dtype: str, num_q_heads: int, num_kv_heads: int, head_size: int,
                q_lens, seq_lens, num_blocks: int | None = None, seed: int = 0,
                pool_factor: float = 1.2, shared_prefix_blocks: int = 0,
                sharing=None) -> StepSpec:
    return StepSpec(name, dtype, num_q_heads, num_kv_heads, head_size,
                    np.asarray(q_lens, np.int64), np.asarray(seq_lens, np.int64),
                    num_blocks=num_blocks, pool_factor=pool_factor,
                    shared_prefix_blocks=shared_prefix_blocks,
                    sharing=None if sharing is None else np.asarray(sharing, bool),
                    seed=seed)


# --------------------------------------------------------------------------
# Generation
# --------------------------------------------------------------------------

def _torch_dtype(dtype: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


def _randn(shape, dtype: torch.dtype, gen: torch.Generator, device) -> torch.Tensor:
    """N(0,1) in fp32, rounded to `dtype` (round to nearest even), generated in
    chunks so that a large bf16 pool needs no full-size fp32 temporary."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    chunk = 1 << 26
    for s in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - s)
        flat[s:s + n] = torch.randn(n, generator=gen, dtype=torch.float32,
                                    device=device).to(dtype)
    return out


def plan_tables(spec: StepSpec):
    """Block tables, pool size and the physical block of every logical block.

    Physical ids come from one seeded permutation of the pool, handed out in
    order: the shared prefix blocks first, then each request's private blocks
    in request order.  Returns (block_tables int32 [B][max_nb], num_blocks,
    unique_blocks)."""
    bs = spec.block_size
    rng = np.random.default_rng(spec.seed + 1000)
    nb = [(-(-int(s) // bs)) for s in spec.seq_lens]
    n_shared = np.zeros(spec.num_seqs, np.int64)
    if spec.shared_prefix_blocks and spec.sharing is not None:
        for r in range(spec.num_seqs):
            if spec.sharing[r]:
                # only full blocks that this step does not write are shared
                hist = int(spec.seq_lens[r] - spec.q_lens[r])
                n_shared[r] = min(spec.shared_prefix_blocks, hist // bs)
    needed = int(sum(nb) - n_shared.sum()) + (spec.shared_prefix_blocks if n_shared.any() else 0)
    num_blocks = spec.num_blocks if spec.num_blocks is not None else int(math.ceil(spec.pool_factor * needed))
    if needed > num_blocks:
        raise ValueError(f"{spec.name}: pool of {num_blocks} blocks < {needed} needed")
    perm = rng.permutation(num_blocks).astype(np.int64)
    cursor = 0
    shared_ids = perm[:spec.shared_prefix_blocks] if n_shared.any() else perm[:0]
    cursor += len(shared_ids)
    max_nb = max(nb) if nb else 1
    bt = np.full((spec.num_seqs, max(max_nb, 1)), -1, dtype=np.int32)
    for r in range(spec.num_seqs):
        k = int(n_shared[r])
        bt[r, :k] = shared_ids[:k]
        own = nb[r] - k
        bt[r, k:nb[r]] = perm[cursor:cursor + own]
        cursor += own
    return bt, num_blocks, needed


@dataclass
class StepMeta:
    """Host metadata of one step (no tensor data)."""
    block_tables: np.ndarray        # int32 [B][max_blocks], -1 past the end
    num_blocks: int
    unique_blocks: int
    query_start_loc: np.ndarray     # int64 [B+1]
    slot_mapping: np.ndarray        # int64 [T]
    hist_mask: np.ndarray           # bool [NB * 16]: slot holds history KV


def make_meta(spec: StepSpec) -> StepMeta:
    """Block tables, query_start_loc, slot_mapping and the history-slot mask."""
    bs = spec.block_size
    B, T = spec.num_seqs, spec.num_tokens
    if np.any(spec.q_lens < 1) or np.any(spec.q_lens > spec.seq_lens):
        raise ValueError("need 1 <= q_len <= seq_len for every request")
    bt, NB, needed = plan_tables(spec)
    qsl = np.zeros(B + 1, np.int64)
    qsl[1:] = np.cumsum(spec.q_lens)
    # slot of each new token: block_table[pos // 16] * 16 + pos % 16
    slot = np.empty(T, np.int64)
    # history slots (filled with data) vs everything else (NaN)
    hist_mask = np.zeros(NB * bs, dtype=bool)
    for r in range(B):
        S, L = int(spec.seq_lens[r]), int(spec.q_lens[r])
        pos = np.arange(S - L, S)
        slot[qsl[r]:qsl[r + 1]] = bt[r, pos // bs].astype(np.int64) * bs + pos % bs
        hpos = np.arange(0, S - L)
        hist_mask[bt[r, hpos // bs].astype(np.int64) * bs + hpos % bs] = True
    if len(np.unique(slot)) != T:
        raise AssertionError("slot_mapping must be unique")
    if np.any(hist_mask[slot]):
        raise AssertionError("a new token's slot holds history")
    return StepMeta(bt, NB, needed, qsl, slot, hist_mask)


def make_step(spec: StepSpec, device="cpu") -> Step:
    """Build all inputs of `spec` on `device`."""
    bs = spec.block_size
    T = spec.num_tokens
    Hq, Hkv, D = spec.num_q_heads, spec.num_kv_heads, spec.head_size
    m = make_meta(spec)
    bt, NB, needed, qsl, slot, hist_mask = (m.block_tables, m.num_blocks, m.unique_blocks,
                                            m.query_start_loc, m.slot_mapping, m.hist_mask)
    dt = _torch_dtype(spec.dtype)
    gen = torch.Generator(device=device)
    gen.manual_seed(spec.seed)
    q = _randn((T, Hq, D), dt, gen, device)
    k = _randn((T, Hkv, D), dt, gen, device)
    v = _randn((T, Hkv, D), dt, gen, device)
    k_cache = _randn((NB, bs, Hkv, D), dt, gen, device)
    v_cache = _randn((NB, bs, Hkv, D), dt, gen, device)
    empty = torch.from_numpy(np.nonzero(~hist_mask)[0]).to(device)
    nan = torch.tensor(float("nan"), dtype=dt, device=device)
    k_cache.view(NB * bs, Hkv, D).index_fill_(0, empty, nan)
    v_cache.view(NB * bs, Hkv, D).index_fill_(0, empty, nan)
    return Step(spec=spec, num_blocks=NB,
                block_tables=torch.from_numpy(bt).to(device),
                seq_lens=torch.from_numpy(spec.seq_lens.astype(np.int32)).to(device),
                query_start_loc=torch.from_numpy(qsl.astype(np.int32)).to(device),
                slot_mapping=torch.from_numpy(slot).to(device),
                q=q, k=k, v=v, k_cache=k_cache, v_cache=v_cache,
                scale=1.0 / math.sqrt(D), unique_blocks=needed)


def make_config(name: str, device="cpu", seed: int | None = None) -> Step:
    fn = CONFIGS[name]
    spec = fn() if seed is None else fn(seed)
    return make_step(spec, device)


def to_numpy_bits(t: torch.Tensor) -> np.ndarray:
    """Raw element bits of a CPU tensor as numpy: bf16 -> uint16, f32 -> float32."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(f"unsupported dtype {t.dtype}")
