"""Shared helpers for the GPU parity tests: run the CUDA path and the oracle
on the same seeded inputs and compare element by element.

Tolerances (bf16 inputs, fp32 accumulation, bf16 or fp32 output):
  max |O - O*|            <= 2e-2
  ||O - O*||_F / ||O*||_F <= 5e-3   (over the whole tensor)
  max |lse - lse*|        <= 1e-3   (rows with a finite reference LSE)
  rows with no visible key: lse = -inf on both sides and O = 0.
"""

import numpy as np
import torch

MAX_ABS = 2e-2
REL_FRO = 5e-3
LSE_ABS = 1e-3


def compare(out, lse, ref_out, ref_lse, rows=None):
    """out/lse: torch (any device); ref_*: numpy float64.  Returns the error dict and asserts the bar."""
    o = out.double().cpu().numpy()
    l = lse.double().cpu().numpy()
    if rows is not None:
        o, l, ref_out, ref_lse = o[rows], l[rows], ref_out[rows], ref_lse[rows]
    fin = np.isfinite(ref_lse)
    err = {
        "max_abs": float(np.abs(o - ref_out).max()) if o.size else 0.0,
        "rel_fro": float(np.linalg.norm(o - ref_out) / max(np.linalg.norm(ref_out), 1e-30)),
        "lse_abs": float(np.abs(l[fin] - ref_lse[fin]).max()) if fin.any() else 0.0,
    }
    assert np.isfinite(o).all(), "non-finite output"
    assert (np.isneginf(l) == ~fin).all(), "-inf LSE rows differ"
    assert not o[~fin].any(), "rows without keys must be zero"
    assert err["max_abs"] <= MAX_ABS, err
    assert err["rel_fro"] <= REL_FRO, err
    assert err["lse_abs"] <= LSE_ABS, err
    return err


def dense_oracle(case, batches=None):
    from oracle import mla_oracle as orc
    return orc.dense_decode(case.q.double().numpy(), case.kv.float().numpy(), case.block_table.numpy(),
                            case.cache_seqlens.numpy(), case.causal, case.scale, batches=batches)


def sparse_oracle(case, batches=None):
    from oracle import mla_oracle as orc
    o, l, bad = orc.sparse_decode(case.q.double().numpy(), case.kv8.numpy(), case.indices.numpy(),
                                  case.topk_length.numpy(), case.scale, batches=batches)
    return o, l


def to_dev(case, dev="cuda"):
    import copy
    c = copy.copy(case)
    for name in ("q", "kv", "kv8", "block_table", "cache_seqlens", "indices", "topk_length"):
        if hasattr(c, name) and getattr(c, name) is not None:
            setattr(c, name, getattr(c, name).to(dev))
    return c
