"""fp64 CPU oracle for one paged-KV attention step.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may call
this module.  The product path never does: it runs the CUDA library and fails
if that library is missing.  This file shares no code with the CUDA path; it
takes plain numpy arrays (bf16 as raw uint16 bits) and does everything in
float64 with textbook formulas, slowly and visibly.

What each function follows:
  blocks_needed     -- "Inside vLLM", section Scheduler (allocate_slots):
                       16 tokens per block, 17 new tokens need ceil(17/16)=2.
  block_bytes       -- "Inside vLLM", section LLM Engine constructor: a block
                       is 2 (K/V) x block_size x num_kv_heads x head_size x
                       dtype bytes.
  slot_of           -- "Serving models at scale with vLLM", section
                       PagedAttention (a block table lists a request's blocks in
                       order) and "Inside vLLM", section Run forward pass
                       (slot_mapping is built while preparing inputs).
  validate_step     -- the invariants the rest relies on.
  cache_write       -- "Inside vLLM", section Prefix Caching (the forward pass
                       fills the allocated blocks with the new tokens' KVs):
                       a byte copy of each new token's K and V into its slot.
  paged_attention   -- "Inside vLLM", section Run forward pass (all sequences
                       flattened into one super-sequence; each token attends
                       only to its own sequence) and "Serving models at scale
                       with vLLM", section Chunked prefill (a later chunk reads
                       the earlier chunks' KV from the cache; a token depends
                       only on the tokens before it).  Softmax attention is
                       written out from its definition.
  within_tolerance,
  error_report      -- the comparison the parity tests apply: the combined
                       elementwise bound |got - ref| <= atol + rtol |ref|, and
                       the absolute and relative errors measured separately
                       (the relative one above a stated |ref| floor).  The pages
                       state no accuracy; the bounds come with the inputs'
                       precision (bf16 in, fp32 accumulate; or fp32).

Readings where the pages are silent (each is stated once more where used):
  * seq_lens[r] counts the KV tokens of request r including this step's new
    tokens; the j-th new token of a chunk of length L sits at position
    S - L + j and attends to positions 0 .. S - L + j (causal).
  * grouped heads: q head h reads kv head h // (Hq / Hkv).
  * cache layout [num_blocks][block_size][Hkv][D], K and V in two arrays.
  * slot_mapping is int64; a negative slot means "do not write this token".
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# Block bookkeeping
# ---------------------------------------------------------------------------

def blocks_needed(num_tokens: int, block_size: int = 16) -> int:
    """Number of KV blocks that hold `num_tokens` tokens: ceil(n / block_size).

    "Inside vLLM", section Scheduler, allocate_slots step 1."""
    if num_tokens < 0 or block_size < 1:
        raise ValueError("num_tokens >= 0 and block_size >= 1 required")
    return (num_tokens + block_size - 1) // block_size


def block_bytes(num_kv_heads: int, head_size: int, dtype_bytes: int, block_size: int = 16) -> int:
    """Bytes of one KV block: 2 (K and V) x block_size x Hkv x D x dtype bytes.

    "Inside vLLM", section LLM Engine constructor."""
    return 2 * block_size * num_kv_heads * head_size * dtype_bytes


def slot_of(block_table_row, position: int, block_size: int = 16) -> int:
    """Physical slot of logical `position`: the block the table names for
    position // block_size, times block_size, plus position % block_size."""
    return int(block_table_row[position // block_size]) * block_size + position % block_size


# ---------------------------------------------------------------------------
# Element widening (bit-exact)
# ---------------------------------------------------------------------------

def widen(x: np.ndarray) -> np.ndarray:
    """Exact float64 value of every element.  uint16 arrays are bf16 bit
    patterns: the bf16 value is the float32 whose upper 16 bits they are."""
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if x.dtype in (np.float32, np.float64):
        return x.astype(np.float64)
    raise TypeError(f"unsupported element type {x.dtype}")


# ---------------------------------------------------------------------------
# Step validation
# ---------------------------------------------------------------------------

def validate_step(block_tables, seq_lens, query_start_loc, num_blocks: int,
                  slot_mapping=None, block_size: int = 16) -> None:
    """Raise ValueError unless the step's metadata is consistent:
    qsl[0] = 0, qsl nondecreasing, 1 <= q_len <= seq_len, the used table
    entries lie in [0, num_blocks), and non-negative slots are unique and
    inside the pool."""
    bt = np.asarray(block_tables)
    S = np.asarray(seq_lens, dtype=np.int64)
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    B = len(S)
    if len(qsl) != B + 1 or qsl[0] != 0:
        raise ValueError("query_start_loc must have B+1 entries starting at 0")
    ql = np.diff(qsl)
    if np.any(ql < 1):
        raise ValueError("every request needs q_len >= 1")
    if np.any(ql > S):
        raise ValueError("q_len must not exceed seq_len")
    for r in range(B):
        used = bt[r, :blocks_needed(int(S[r]), block_size)]
        if np.any(used < 0) or np.any(used >= num_blocks):
            raise ValueError(f"request {r}: block id outside the pool")
    if slot_mapping is not None:
        sm = np.asarray(slot_mapping, dtype=np.int64)
        if len(sm) != qsl[-1]:
            raise ValueError("slot_mapping needs one entry per new token")
        live = sm[sm >= 0]
        if np.any(live >= num_blocks * block_size):
            raise ValueError("slot outside the pool")
        if len(np.unique(live)) != len(live):
            raise ValueError("two tokens write one slot")


# ---------------------------------------------------------------------------
# reshape_and_cache: the slot write
# ---------------------------------------------------------------------------

def cache_write(k, v, slot_mapping, k_cache, v_cache, block_size: int = 16):
    """Return copies of the caches with token t's K/V copied, element bits
    unchanged, to slot s = slot_mapping[t]: block s // block_size, row
    s % block_size.  Tokens with s < 0 are skipped.

    k, v: [T][Hkv][D]; caches: [NB][block_size][Hkv][D]."""
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    for t, s in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if s < 0:
            continue
        kc[s // block_size, s % block_size] = k[t]
        vc[s // block_size, s % block_size] = v[t]
    return kc, vc


# ---------------------------------------------------------------------------
# Attention over the flattened super-sequence
# ---------------------------------------------------------------------------

def gather_request_kv(cache, block_table_row, seq_len: int, kv_head: int,
                      block_size: int = 16) -> np.ndarray:
    """Logical rows 0 .. seq_len-1 of one request and kv head, as float64
    [seq_len][D]: position p lives in block table[p // bs], row p % bs."""
    p = np.arange(seq_len)
    phys = np.asarray(block_table_row)[p // block_size].astype(np.int64)
    return widen(cache[phys, p % block_size, kv_head, :])


def paged_attention(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc,
                    scale: float, num_kv_heads: int, block_size: int = 16,
                    requests=None) -> np.ndarray:
    """fp64 attention output [T][Hq][D] for every new token.

    Request r owns flattened rows qsl[r] .. qsl[r+1]-1 (L = q_len rows) and
    S = seq_lens[r] KV positions.  Row j is at position S - L + j and, for q
    head h with kv head g = h // (Hq / Hkv):
        x_p = scale * sum_d q[d] * K[p][d]            for p = 0 .. S - L + j
        o   = sum_p exp(x_p - max x) V[p] / sum_p exp(x_p - max x)
    Rows of requests not in `requests` (if given) are left NaN."""
    qf = widen(np.asarray(q))
    T, Hq, D = qf.shape
    if Hq % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    G = Hq // num_kv_heads
    S_all = np.asarray(seq_lens, dtype=np.int64)
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    out = np.full((T, Hq, D), np.nan)
    todo = range(len(S_all)) if requests is None else requests
    for r in todo:
        S = int(S_all[r])
        t0, t1 = int(qsl[r]), int(qsl[r + 1])
        L = t1 - t0
        for g in range(num_kv_heads):
            K = gather_request_kv(k_cache, block_tables[r], S, g, block_size)
            V = gather_request_kv(v_cache, block_tables[r], S, g, block_size)
            for j in range(L):
                pos = S - L + j
                for h in range(g * G, (g + 1) * G):
                    x = scale * (K[:pos + 1] @ qf[t0 + j, h])
                    w = np.exp(x - x.max())
                    out[t0 + j, h] = (w @ V[:pos + 1]) / w.sum()
    return out


def paged_attention_rows(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc,
                         scale: float, num_kv_heads: int, rows, block_size: int = 16):
    """The same definition as `paged_attention`, for a list of (token t, q head h)
    pairs only; returns float64 [len(rows)][D].  Used to check sampled outputs of
    workloads too large to evaluate whole."""
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    S_all = np.asarray(seq_lens, dtype=np.int64)
    Hq = q.shape[1]
    G = Hq // num_kv_heads
    res = []
    for t, h in rows:
        r = int(np.searchsorted(qsl, t, side="right") - 1)
        S, L = int(S_all[r]), int(qsl[r + 1] - qsl[r])
        pos = S - L + (t - int(qsl[r]))
        g = h // G
        K = gather_request_kv(k_cache, block_tables[r], pos + 1, g, block_size)
        V = gather_request_kv(v_cache, block_tables[r], pos + 1, g, block_size)
        x = scale * (K @ widen(np.asarray(q[t, h])))
        w = np.exp(x - x.max())
        res.append((w @ V) / w.sum())
    return np.array(res)


def within_tolerance(got, ref, atol: float, rtol: float):
    """Elementwise |got - ref| <= atol + rtol * |ref|, with both sides finite
    (an infinite ref would otherwise admit any got); returns (ok, max_abs,
    max_rel over |ref| > 1e-2)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    ok = bool(np.all(np.isfinite(got) & np.isfinite(ref) & (err <= atol + rtol * np.abs(ref))))
    big = np.abs(ref) > 1e-2
    max_rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    return ok, float(err.max()) if err.size else 0.0, max_rel


def error_report(got, ref, rel_floor: float) -> dict:
    """The two error measures of the stated accuracy target, each on its own.

      nonfinite  number of elements of `got` that are NaN or infinite
      max_abs    max |got - ref| over every element (inf when any element of
                 got or ref is not finite, so a NaN can never pass a bound)
      max_rel    max |got - ref| / |ref| over the elements with
                 |ref| >= rel_floor (0 when there are none)
      rel_count  how many elements max_rel was taken over

    A relative error has no meaning where ref is 0, so it is measured only
    above a stated floor; below it the absolute bound alone applies."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if got.shape != ref.shape:
        raise ValueError(f"shapes differ: {got.shape} vs {ref.shape}")
    finite = np.isfinite(got) & np.isfinite(ref)
    err = np.abs(got - ref)
    if not finite.all():
        max_abs = float("inf")
    else:
        max_abs = float(err.max()) if err.size else 0.0
    big = np.abs(ref) >= rel_floor
    if big.any():
        rel = np.where(finite[big], err[big] / np.abs(ref[big]), np.inf)
        max_rel = float(rel.max())
    else:
        max_rel = 0.0
    return {"nonfinite": int((~np.isfinite(got)).sum()), "max_abs": max_abs,
            "max_rel": max_rel, "rel_count": int(big.sum()), "rel_floor": float(rel_floor)}
