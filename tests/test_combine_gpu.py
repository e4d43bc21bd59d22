"""The split combine (mla_combine) on hand-made partials, against the
oracle's merge (combine_partials: the LSE rule of FlashMLA PR #183,
Summary), through the C ABI on the GPU.

Each case fixes a split_offset by hand, so that every layout the host can
pick is exercised: whole-row warps (>= 8192 rows), split-parallel blocks
(units averaging 8 or more splits) and the streaming kernel (the rest), with
units of 0 splits (out 0, lse -inf), 1 split (left alone), several splits,
more than 32 splits, and rows whose splits are all empty.  A split with lse
-inf holds NaN in its partial row: it must weigh exactly 0."""

import numpy as np
import pytest
import torch

import mla_paged_kv_gb300 as mla
from oracle import mla_oracle as orc

pytestmark = pytest.mark.gpu

SENTINEL = 7.25  # written into out before the call: units with one split keep it


def build_case(splits, rows, num_parts, seed, empty_frac=0.15):
    n_units = len(splits)
    so = np.concatenate([[0], np.cumsum(splits)]).astype(np.int32)
    slots = n_units + num_parts
    assert so[-1] <= slots
    rng = np.random.default_rng(seed)
    O = rng.standard_normal((slots, rows, 512)).astype(np.float32)
    L = (3.0 * rng.standard_normal((slots, rows))).astype(np.float32)
    L[rng.random((slots, rows)) < empty_frac] = -np.inf
    # the first row of every multi-split unit: all its splits empty
    for u in range(n_units):
        if splits[u] >= 2:
            L[so[u]:so[u + 1], 0] = -np.inf
    O_dev = O.copy()
    O_dev[np.isneginf(L)] = np.nan           # whatever an empty split's partial holds
    O[np.isneginf(L)] = 0.0                  # the oracle's input: weight 0 anyway
    return so, O, L, O_dev


def run_combine(so, O_dev, L, n_units, rows, num_parts, out_dtype):
    nbytes = mla.mla_workspace_bytes(n_units, rows, num_parts)
    o_bytes = O_dev.nbytes
    lse_off = (o_bytes + 255) // 256 * 256
    ws = np.zeros(nbytes, dtype=np.uint8)
    ws[:o_bytes] = O_dev.reshape(-1).view(np.uint8)
    ws[lse_off:lse_off + L.nbytes] = L.reshape(-1).view(np.uint8)
    ws_d = torch.from_numpy(ws).cuda()
    so_d = torch.from_numpy(so).cuda()
    out = torch.full((n_units, rows, 512), SENTINEL, dtype=out_dtype, device="cuda")
    lse = torch.full((n_units, rows), SENTINEL, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_combine(ws_d, so_d, n_units, rows, num_parts, out, lse, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def check(so, O, L, out, lse, out_dtype):
    rel = 0.0 if out_dtype == torch.float32 else 2.0 ** -8   # bf16: within one ulp of the merge
    for u in range(len(so) - 1):
        n = so[u + 1] - so[u]
        if n == 1:
            assert (out[u] == SENTINEL).all() and (lse[u] == SENTINEL).all(), u
            continue
        if n == 0:
            assert (out[u] == 0).all() and np.isneginf(lse[u]).all(), u
            continue
        parts = [(O[s].astype(np.float64), L[s].astype(np.float64)) for s in range(so[u], so[u + 1])]
        ro, rl = orc.combine_partials(parts)
        assert np.isfinite(out[u]).all(), u
        err = np.abs(out[u] - ro) - rel * np.abs(ro)
        assert err.max() <= 2e-5, (u, err.max())
        fin = np.isfinite(rl)
        assert (np.isneginf(lse[u]) == ~fin).all(), u
        assert not out[u][~fin].any(), u
        assert np.abs(lse[u][fin] - rl[fin]).max() <= 1e-5, u


SEEDS = {"whole_rows": 11, "split_parallel": 12, "stream": 13, "stream_ragged": 14}
CASES = {
    # 64 units x 128 rows = 8192 rows: whole-row warps
    "whole_rows": (lambda: [2] * 20 + [1] * 10 + [3] * 10 + [0] * 4 + [2] * 20, 128, 76),
    # few rows, many splits per unit: split-parallel blocks
    "split_parallel": (lambda: [40, 9, 1, 0, 12], 64, 76),
    # the rest: the streaming kernel (one item = 16 rows), with a unit of 40 splits
    "stream": (lambda: [3, 2, 1, 0, 40, 5, 2, 2, 3, 1, 4, 2], 256, 76),
    # streaming kernel, rows not a multiple of 16 (a partial last item)
    "stream_ragged": (lambda: [2, 3, 1, 6, 0, 2], 40, 20),
}


@pytest.mark.parametrize("layout", sorted(CASES))
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_combine_matches_the_oracle_merge(layout, out_dtype):
    mk, rows, num_parts = CASES[layout]
    splits = mk()
    n_units = len(splits)
    so, O, L, O_dev = build_case(splits, rows, num_parts, seed=SEEDS[layout])
    # the host's choice of layout, restated so that the case really covers it
    whole = n_units * rows >= 8192
    split_par = not whole and num_parts >= 8 * n_units
    assert {"whole_rows": whole, "split_parallel": split_par}.get(layout, not whole and not split_par)
    out, lse = run_combine(so, O_dev, L, n_units, rows, num_parts, out_dtype)
    check(so, O, L, out, lse, out_dtype)


def test_combine_layouts_agree_bit_for_bit():
    """The whole-row and streaming kernels run the same arithmetic in the
    same order: the same units merged under either layout give the same bits
    (here the streaming layout is reached by passing fewer rows per unit,
    i.e. the first 64 rows of each unit's partials)."""
    splits = [2, 3, 5, 2] * 16
    rows, parts = 128, 128                                   # 192 splits in 192 slots
    so, O, L, O_dev = build_case(splits, rows, parts, seed=5)
    out_w, lse_w = run_combine(so, O_dev, L, len(splits), rows, parts, torch.float32)
    # the same partial rows 0..63 of every slot, laid out with rows = 64
    so2, O2, L2, O2_dev = so, np.ascontiguousarray(O[:, :64]), np.ascontiguousarray(L[:, :64]), \
        np.ascontiguousarray(O_dev[:, :64])
    out_s, lse_s = run_combine(so2, O2_dev, L2, len(splits), 64, parts, torch.float32)
    assert np.array_equal(out_w[:, :64], out_s) and np.array_equal(lse_w[:, :64], lse_s)
