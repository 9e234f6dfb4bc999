"""Test helpers: run one step through libpa (GPU) and through the oracle (CPU)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_attention_04_gb300 as P
from paged_kv_attention_04_gb300 import workloads as W

# (max-abs, max-rel) error bounds: bf16 in with fp32 accumulation, and fp32
TOL = {"bf16": (1e-2, 2e-2), "f32": (1e-5, 1e-5)}
# |ref| from which the relative error is gated (below it, max-abs alone).
# bf16: half of atol / rtol = 0.5, the |ref| above which the relative bound is
# already implied by the absolute one.  Below 0.25 the bf16 rounding of the
# softmax weights that enter the P.V product (relative 2^-9 each) leaves
# relative errors of 2-4e-2 on rows of few keys even with exact fp32 arithmetic
# elsewhere.  fp32: the accumulated rounding of exp2 and the dot products
# stays under 1e-5 relative from |ref| = 0.05 on.
REL_FLOOR = {"bf16": 0.25, "f32": 0.05}


def bits(t: torch.Tensor) -> np.ndarray:
    return W.to_numpy_bits(t)


def raw_bits(t: torch.Tensor) -> np.ndarray:
    """Element bits as unsigned integers (NaN payloads compare exactly)."""
    a = W.to_numpy_bits(t)
    return a.view(np.uint32) if a.dtype == np.float32 else a


def run_gpu(step: W.Step, sentinel: float = float("nan")):
    """pa_cache_write then pa_forward on copies of the caches.  Returns
    (out, k_cache, v_cache, status)."""
    kc = step.k_cache.clone()
    vc = step.v_cache.clone()
    lay = P.layout_of(kc, step.spec.num_q_heads)
    status = torch.zeros(1, dtype=torch.int32, device=kc.device)
    P.pa_cache_write(step.k, step.v, step.slot_mapping, kc, vc, lay, status)
    ws = P.alloc_workspace(lay, step.spec.num_seqs, step.spec.num_tokens, step.max_seq_len,
                           device=kc.device)
    out = torch.full_like(step.q, sentinel)
    P.pa_forward(step.q, kc, vc, step.block_tables, step.seq_lens, step.query_start_loc,
                 step.max_query_len, step.max_seq_len, step.scale, out, ws, lay, status)
    torch.cuda.synchronize()
    return out, kc, vc, int(status.item())


def run_oracle(step: W.Step):
    """The oracle's slot write and fp64 attention on the step's (CPU) tensors."""
    kc, vc = oracle.cache_write(bits(step.k), bits(step.v), step.slot_mapping.cpu().numpy(),
                                bits(step.k_cache), bits(step.v_cache))
    out = oracle.paged_attention(bits(step.q), kc, vc, step.block_tables.cpu().numpy(),
                                 step.seq_lens.cpu().numpy(), step.query_start_loc.cpu().numpy(),
                                 step.scale, step.spec.num_kv_heads)
    return out, kc, vc


def assert_close(got: torch.Tensor, ref: np.ndarray, dtype: str, what: str = ""):
    """The parity gates, all of which must hold:
      * every output element is finite;
      * combined, per element: |got - ref| <= atol + rtol |ref|;
      * max-abs error <= atol over every element;
      * max-rel error <= rtol over the elements with |ref| >= REL_FLOOR[dtype].
    Returns (max_abs, max_rel)."""
    atol, rtol = TOL[dtype]
    g = oracle.widen(bits(got)) if got.dtype == torch.bfloat16 else got.detach().cpu().double().numpy()
    ok, _, _ = oracle.within_tolerance(g, ref, atol, rtol)
    rep = oracle.error_report(g, ref, REL_FLOOR[dtype])
    msg = (f"{what}: max_abs={rep['max_abs']:.3g} (gate {atol:g}), max_rel={rep['max_rel']:.3g} "
           f"over |ref| >= {REL_FLOOR[dtype]:g} (gate {rtol:g}), nonfinite={rep['nonfinite']}")
    if rep["nonfinite"]:
        raise AssertionError(f"non-finite outputs; {msg}")
    if not ok:
        err = np.abs(g - ref)
        bad = np.argwhere(~(err <= atol + rtol * np.abs(ref)))
        raise AssertionError(f"{len(bad)} elements outside atol + rtol|ref|; first "
                             f"{bad[:5].tolist()}; {msg}")
    if not rep["max_abs"] <= atol:
        raise AssertionError(f"max_abs above its gate; {msg}")
    if not rep["max_rel"] <= rtol:
        raise AssertionError(f"max_rel above its gate; {msg}")
    return rep["max_abs"], rep["max_rel"]
