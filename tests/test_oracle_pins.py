"""Pins for the CPU oracle, independent of the oracle's own code.

Every check here compares the oracle with something it does not share code
with: torch's scaled_dot_product_attention in float64 (a different library
route, fed by a separate gather), closed-form results, invariants of the
mathematics, torch's own FP8/bf16 conversions, and the sizes the pages print.
A plausible mistake in the oracle (a dropped RoPE term, a transposed operand,
a wrong scale, an off-by-one causal offset, log2 instead of ln, a wrong
record offset or scale group) fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import mla_oracle as orc
from mla_paged_kv_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TOL = 1e-12


# ---------------------------------------------------------------- helpers

def f64(t):
    return t.double().numpy()


def sdpa_dense_reference(case, b):
    """torch fp64 SDPA over keys gathered with torch indexing + explicit causal bias."""
    L = int(case.cache_seqlens[b])
    flat = case.kv.double().reshape(-1, 576)
    j = torch.arange(L)
    slot = case.block_table[b].long()[j // 64] * 64 + (j % 64)
    K = flat[slot]                                   # [L, 576]
    V = K[:, :512]
    s_q, h_q = case.s_q, case.h_q
    q = case.q[b].double().reshape(s_q * h_q, 576)
    tok = torch.arange(s_q * h_q) // h_q
    if case.causal:
        allowed = j[None, :] <= (L - s_q + tok[:, None])
    else:
        allowed = torch.ones(s_q * h_q, L, dtype=torch.bool)
    bias = torch.zeros(s_q * h_q, L, dtype=torch.float64).masked_fill(~allowed, float("-inf"))
    out = torch.nn.functional.scaled_dot_product_attention(
        q[None], K[None], V[None], attn_mask=bias[None], scale=case.scale)[0]
    lse = torch.logsumexp(q @ K.T * case.scale + bias, dim=-1)
    return out.numpy().reshape(s_q, h_q, 512), lse.numpy().reshape(s_q, h_q)


def torch_decode_records(kv8, slots):
    """Decode records with torch's own fp8/bf16 conversions (float64 result)."""
    rec = kv8.reshape(-1, 656)[slots.long()]
    codes = rec[:, :512].contiguous().view(torch.float8_e4m3fn).double()
    scales = rec[:, 512:528].contiguous().view(torch.float32).double()       # [n, 4]
    rope = rec[:, 528:656].contiguous().view(torch.bfloat16).double()        # [n, 64]
    nope = (codes.reshape(-1, 4, 128) * scales[:, :, None]).reshape(-1, 512)
    return torch.cat([nope, rope], dim=1)


def dense_by_hand(q, keys, scale, L=None, causal=False, s_q=1, h_q=None):
    """Build a one-request case from explicit key rows (block table = identity)."""
    n = keys.shape[0]
    pages = max(1, (n + 63) // 64)
    kv = np.zeros((pages, 64, 576))
    kv.reshape(-1, 576)[:n] = keys
    bt = np.arange(pages, dtype=np.int32)[None]
    out, lse = orc.dense_decode(q[None], kv, bt, np.array([n if L is None else L]), causal, scale)
    return out[0], lse[0]


# ---------------------------------------------------------------- number formats

def test_e4m3_exhaustive_against_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3fn_to_f64(codes)
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    nan_ours, nan_ref = np.isnan(ours), np.isnan(ref)
    assert (nan_ours == nan_ref).all()
    assert set(np.nonzero(nan_ours)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan_ours], ref[~nan_ref])


def test_e4m3_closed_forms():
    # s eeee mmm with bias 7: values fixed by the format definition itself
    cases = {0x00: 0.0, 0x38: 1.0, 0xC0: -2.0, 0x3C: 1.5, 0x7E: 448.0, 0xFE: -448.0,
             0x08: 2.0 ** -6, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x30: 0.5}
    got = orc.e4m3fn_to_f64(np.array(list(cases), dtype=np.uint8))
    assert got.tolist() == list(cases.values())


def test_bf16_bits_against_torch():
    g = torch.Generator().manual_seed(7)
    x = (torch.randn(4096, generator=g) * 100).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.bf16_bits_to_f64(bits), x.double().numpy())


# ---------------------------------------------------------------- sizes printed by the pages

def test_page_printed_sizes_pin_layout_constants():
    facts = json.load(open(os.path.join(GOLDEN, "page_facts.json")))
    tok_bytes = orc.D_QK * 2                                     # bf16 latent row
    f = facts["dense_kv_bytes_b64_sk4096"]
    assert round(f["batch"] * f["seqlen"] * tok_bytes / 1e6) == f["value_mb"]
    f = facts["sq_tile_bytes_16_rows"]
    assert f["rows"] * tok_bytes / 1024 == f["value_kb"]
    f = facts["sk_page_bytes"]
    assert f["tokens"] * tok_bytes / 1024 == f["value_kb"] and f["tokens"] == orc.PAGE_SIZE
    f = facts["sk_16tok_3stage_bytes"]
    assert f["tokens"] * f["stages"] * tok_bytes / 1024 == f["value_kb"]
    f = facts["packed_workspace_per_row_topk2048"]
    assert round(f["topk"] * orc.RECORD_BYTES / 2 ** 20, 3) == f["value_mib"]
    f = facts["record_parts_bytes"]
    assert (f["nope"], f["scales"], f["rope"]) == (orc.NOPE_BYTES, orc.ROPE_OFF - orc.SCALE_OFF,
                                                    orc.RECORD_BYTES - orc.ROPE_OFF)
    assert f["nope"] + f["scales"] + f["rope"] == orc.RECORD_BYTES
    assert f["scales"] // 4 * orc.GROUP == orc.NOPE_BYTES        # one fp32 scale per 128 codes


def test_record_decode_by_hand():
    rec = np.zeros(656, dtype=np.uint8)
    rec[0], rec[1], rec[127] = 0x38, 0xC0, 0x7E          # 1, -2, 448 (group 0)
    rec[128], rec[255] = 0x3C, 0x01                      # 1.5, 2^-9 (group 1)
    rec[256], rec[511] = 0x30, 0x08                      # 0.5 (group 2), 2^-6 (group 3)
    rec[512:528] = np.array([0.5, 2.0, 4.0, 0.25], dtype="<f4").view(np.uint8)
    rope = np.zeros(64, dtype="<u2")
    rope[0], rope[63] = 0x3FC0, 0xBF80                   # bf16 1.5, -1.0
    rec[528:656] = rope.view(np.uint8)
    k = orc.decode_record(rec)
    expect = np.zeros(576)
    expect[0], expect[1], expect[127] = 0.5, -1.0, 224.0
    expect[128], expect[255] = 3.0, 2.0 ** -8
    expect[256], expect[511] = 2.0, 2.0 ** -8
    expect[512], expect[575] = 1.5, -1.0
    assert np.array_equal(k, expect)


def test_unpack_bit_exact_against_torch():
    case = wl.sparse_case(2, 1, 8, topk=64, pages_per_req=2, topk_lo=40, topk_hi=64, seed=11)
    idx = case.indices.reshape(-1)
    ours, bad = orc.unpack_records(case.kv8.numpy(), idx.numpy())
    assert bad == 0
    valid = idx >= 0
    rec = case.kv8.reshape(-1, 656)[idx[valid].long()]
    codes = rec[:, :512].contiguous().view(torch.float8_e4m3fn).float()
    sc = rec[:, 512:528].contiguous().view(torch.float32)
    nope = (codes.reshape(-1, 4, 128) * sc[:, :, None]).reshape(-1, 512)        # fp32 multiply
    rope = rec[:, 528:].contiguous().view(torch.bfloat16).float()
    ref = torch.cat([nope, rope], 1).numpy()
    assert np.array_equal(ours[valid.numpy()].view(np.uint32), ref.view(np.uint32))
    assert not ours[~valid.numpy()].any()


# ---------------------------------------------------------------- brute force vs torch SDPA

@pytest.mark.parametrize("s_q,h_q,causal", [(1, 16, False), (2, 8, True), (2, 4, False), (1, 4, True)])
@pytest.mark.parametrize("lens", [(1, 63), (64, 65), (130, 200)])
def test_dense_matches_torch_sdpa(s_q, h_q, causal, lens):
    case = wl.dense_case(2, s_q, h_q, 0, seqlens=lens, causal=causal, seed=sum(lens) + s_q)
    out, lse = orc.dense_decode(f64(case.q), f64(case.kv), case.block_table.numpy(),
                                case.cache_seqlens.numpy(), case.causal, case.scale)
    for b in range(2):
        if causal and int(case.cache_seqlens[b]) < s_q:
            continue          # rows with no visible key: covered by a closed-form test
        ro, rl = sdpa_dense_reference(case, b)
        assert np.abs(out[b] - ro).max() < TOL
        assert np.abs(lse[b] - rl).max() < TOL


def test_dense_peaky_matches_torch_sdpa():
    case = wl.dense_case(1, 1, 16, 0, seqlens=[150], q_scale=8.0, seed=5)
    out, lse = orc.dense_decode(f64(case.q), f64(case.kv), case.block_table.numpy(),
                                case.cache_seqlens.numpy(), False, case.scale)
    ro, rl = sdpa_dense_reference(case, 0)
    assert np.abs(out[0] - ro).max() < TOL and np.abs(lse[0] - rl).max() < TOL


def test_sparse_matches_torch_sdpa():
    case = wl.sparse_case(2, 2, 8, topk=64, pages_per_req=4, topk_lo=20, topk_hi=64, seed=3)
    ind = case.indices.clone()
    ind[0, 0, 3] = -1                      # -1 inside the valid prefix
    ind[1, 1, 5] = ind[1, 1, 2]            # a duplicated index
    tl = case.topk_length
    out, lse, bad = orc.sparse_decode(f64(case.q), case.kv8.numpy(), ind.numpy(), tl.numpy(), case.scale)
    assert bad == 0
    for b in range(2):
        for i in range(2):
            t = torch.arange(64)
            keep = (t < int(tl[b, i])) & (ind[b, i] != -1)
            K = torch_decode_records(case.kv8, ind[b, i][keep])
            q = case.q[b, i].double()
            ro = torch.nn.functional.scaled_dot_product_attention(
                q[None], K[None], K[None, :, :512], scale=case.scale)[0]
            rl = torch.logsumexp(q @ K.T * case.scale, dim=-1)
            assert np.abs(out[b, i] - ro.numpy()).max() < TOL
            assert np.abs(lse[b, i] - rl.numpy()).max() < TOL


# ---------------------------------------------------------------- closed forms

def _rng(seed):
    return np.random.default_rng(seed)


def test_single_key_gives_its_value():
    r = _rng(1)
    k = r.standard_normal((1, 576))
    q = r.standard_normal((1, 3, 576))
    out, lse = dense_by_hand(q, k, 0.1)
    assert np.allclose(out[0], np.broadcast_to(k[0, :512], (3, 512)), rtol=0, atol=TOL)
    assert np.allclose(lse[0], 0.1 * (q[0] @ k[0]), rtol=0, atol=TOL)


def test_identical_keys_give_value_and_log_n():
    r = _rng(2)
    n = 77
    k = np.repeat(r.standard_normal((1, 576)), n, axis=0)
    q = r.standard_normal((1, 2, 576))
    out, lse = dense_by_hand(q, k, 1 / 24)
    assert np.allclose(out[0], k[0, :512], rtol=0, atol=TOL)
    assert np.allclose(lse[0], (q[0] @ k[0]) / 24 + math.log(n), rtol=0, atol=TOL)


def test_equal_scores_give_mean_of_values():
    r = _rng(3)
    n = 90
    k = r.standard_normal((n, 576))
    k[:, 512:] = r.standard_normal(64)               # shared RoPE part
    q = np.zeros((1, 4, 576))
    q[0, :, 512:] = r.standard_normal((4, 64))       # q only sees the RoPE part
    out, lse = dense_by_hand(q, k, 0.3)
    assert np.allclose(out[0], k[:, :512].mean(axis=0), rtol=0, atol=TOL)
    assert np.allclose(lse[0], 0.3 * (q[0, :, 512:] @ k[0, 512:]) + math.log(n), rtol=0, atol=TOL)


def test_zero_query_gives_plain_average():
    r = _rng(4)
    n = 129
    k = r.standard_normal((n, 576))
    out, lse = dense_by_hand(np.zeros((1, 2, 576)), k, 1 / 24)
    assert np.allclose(out[0], k[:, :512].mean(axis=0), rtol=0, atol=TOL)
    assert np.allclose(lse[0], math.log(n), rtol=0, atol=TOL)


def test_two_keys_logistic_weights():
    r = _rng(5)
    k = r.standard_normal((2, 576))
    q = r.standard_normal((1, 1, 576))
    s = 0.2 * (q[0, 0] @ k.T)
    w0 = 1 / (1 + math.exp(s[1] - s[0]))
    out, lse = dense_by_hand(q, k, 0.2)
    assert np.allclose(out[0, 0], w0 * k[0, :512] + (1 - w0) * k[1, :512], rtol=0, atol=TOL)
    assert abs(lse[0, 0] - (max(s) + math.log1p(math.exp(min(s) - max(s))))) < TOL


def test_weights_sum_to_one():
    r = _rng(6)
    k = r.standard_normal((300, 576))
    k[:, 7] = 1.0
    q = r.standard_normal((1, 5, 576)) * 3
    out, _ = dense_by_hand(q, k, 1 / 24)
    assert np.abs(out[0, :, 7] - 1.0).max() < TOL


def test_causal_row_with_no_visible_key():
    r = _rng(7)
    k = r.standard_normal((1, 576))
    q = r.standard_normal((1, 2, 576))
    q = q.reshape(2, 1, 576)[None, :, :, :]                 # s_q=2, h_q=1
    kv = np.zeros((1, 64, 576))
    kv[0, 0] = k[0]
    out, lse = orc.dense_decode(q, kv, np.zeros((1, 1), np.int32), np.array([1]), True, 0.5)
    assert not out[0, 0].any() and lse[0, 0, 0] == -np.inf  # token 0 sees j <= -1
    assert np.allclose(out[0, 1, 0], k[0, :512], atol=TOL)   # token 1 sees key 0


def test_empty_request_and_empty_sparse_selection():
    case = wl.dense_case(2, 1, 4, 0, seqlens=[0, 5], seed=9)
    out, lse = orc.dense_decode(f64(case.q), f64(case.kv), case.block_table.numpy(),
                                case.cache_seqlens.numpy(), False, case.scale)
    assert not out[0].any() and np.isneginf(lse[0]).all() and np.isfinite(lse[1]).all()
    sc = wl.sparse_case(1, 1, 4, topk=64, pages_per_req=2, topk_lengths=[[0]], seed=9)
    o, l, _ = orc.sparse_decode(f64(sc.q), sc.kv8.numpy(), sc.indices.numpy(), sc.topk_length.numpy(), sc.scale)
    assert not o.any() and np.isneginf(l).all()
    ind = sc.indices.clone()
    ind[:] = -1
    o, l, _ = orc.sparse_decode(f64(sc.q), sc.kv8.numpy(), ind.numpy(), None, sc.scale)
    assert not o.any() and np.isneginf(l).all()


def test_bad_index_is_masked_and_counted():
    sc = wl.sparse_case(1, 1, 4, topk=64, pages_per_req=2, topk_lengths=[[64]], seed=10)
    ind = sc.indices.clone()
    good, _, _ = orc.sparse_decode(f64(sc.q), sc.kv8.numpy(), np.where(np.arange(64) == 5, -1, ind.numpy()),
                                   None, sc.scale)
    ind[0, 0, 5] = sc.kv8.shape[0] * 64       # one past the pool
    out, lse, bad = orc.sparse_decode(f64(sc.q), sc.kv8.numpy(), ind.numpy(), None, sc.scale)
    assert bad == 1 and np.array_equal(out, good)


# ---------------------------------------------------------------- invariants

def test_split_combine_equals_unsplit():
    r = _rng(8)
    for trial in range(6):
        n = int(r.integers(1, 400))
        keys = r.standard_normal((n, 576))
        q = r.standard_normal((12, 576)) * (8 if trial % 2 else 1)
        full_o, full_l = orc.attend(q, keys, 1 / 24)
        cuts = sorted(set([0, n] + r.integers(0, n + 1, size=int(r.integers(0, 6))).tolist()))
        cuts = [0] + cuts[1:-1] + [cuts[-1]]
        cuts.insert(1, 0)                                  # force one empty split
        parts = orc.split_partials(q, keys, 1 / 24, cuts)
        o, l = orc.combine_partials(parts)
        assert np.abs(o - full_o).max() < TOL and np.abs(l - full_l).max() < TOL


def test_block_table_permutation_is_bit_identical():
    case = wl.dense_case(3, 2, 4, 0, seqlens=[70, 129, 5], causal=True, seed=12)
    args = (f64(case.q), f64(case.kv), case.block_table.numpy(), case.cache_seqlens.numpy(), True, case.scale)
    o1, l1 = orc.dense_decode(*args)
    P = case.kv.shape[0]
    perm = np.random.default_rng(1).permutation(P)
    kv2 = np.empty_like(args[1])
    kv2[perm] = args[1]
    bt = case.block_table.numpy()
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    o2, l2 = orc.dense_decode(args[0], kv2, bt2, args[3], True, case.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_poison_in_unused_slots_is_bit_identical():
    case = wl.dense_case(2, 1, 8, 0, seqlens=[70, 33], seed=13)
    kv = f64(case.kv)
    o1, l1 = orc.dense_decode(f64(case.q), kv, case.block_table.numpy(), case.cache_seqlens.numpy(), False, case.scale)
    used = np.zeros(kv.shape[:2], bool)
    for b in range(2):
        L = int(case.cache_seqlens[b])
        for j in range(L):
            used[int(case.block_table[b, j // 64]), j % 64] = True
    kv2 = np.where(used[:, :, None], kv, -7.0e2)
    o2, l2 = orc.dense_decode(f64(case.q), kv2, case.block_table.numpy(), case.cache_seqlens.numpy(), False, case.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_causally_hidden_key_does_not_reach_token0():
    case = wl.dense_case(1, 2, 4, 0, seqlens=[100], causal=True, seed=14)
    kv = f64(case.kv)
    o1, l1 = orc.dense_decode(f64(case.q), kv, case.block_table.numpy(), case.cache_seqlens.numpy(), True, case.scale)
    page = int(case.block_table[0, 99 // 64])
    kv[page, 99 % 64] += 3.0                 # the last key: only token 1 may see it
    o2, l2 = orc.dense_decode(f64(case.q), kv, case.block_table.numpy(), case.cache_seqlens.numpy(), True, case.scale)
    assert np.array_equal(o1[0, 0], o2[0, 0]) and np.array_equal(l1[0, 0], l2[0, 0])
    assert not np.array_equal(o1[0, 1], o2[0, 1])


def test_sparse_reversal_and_unselected_records():
    sc = wl.sparse_case(1, 1, 8, topk=128, pages_per_req=4, topk_lengths=[[128]], seed=15)
    ind = sc.indices.clone()
    ind[0, 0, ::7] = -1
    q = f64(sc.q)
    o1, l1, _ = orc.sparse_decode(q, sc.kv8.numpy(), ind.numpy(), None, sc.scale)
    o2, l2, _ = orc.sparse_decode(q, sc.kv8.numpy(), ind.flip(-1).numpy(), None, sc.scale)
    assert np.abs(o1 - o2).max() < TOL and np.abs(l1 - l2).max() < TOL
    kv8 = sc.kv8.clone().reshape(-1, 656)
    chosen = torch.zeros(kv8.shape[0], dtype=torch.bool)
    chosen[ind[ind >= 0].long()] = True
    kv8[~chosen, :512] = 0x7E                # 448 in every unselected record
    o3, l3, _ = orc.sparse_decode(q, kv8.reshape(sc.kv8.shape).numpy(), ind.numpy(), None, sc.scale)
    assert np.array_equal(o1, o3) and np.array_equal(l1, l3)


def test_sparse_topk_length_prefix():
    sc = wl.sparse_case(1, 1, 4, topk=64, pages_per_req=2, topk_lengths=[[30]], seed=16)
    q = f64(sc.q)
    ind = sc.indices.clone()
    full = torch.cat([ind[0, 0, :30], torch.full((34,), -1, dtype=torch.int32)])
    o1, l1, _ = orc.sparse_decode(q, sc.kv8.numpy(), full.reshape(1, 1, 64).numpy(), None, sc.scale)
    ind[0, 0, 30:] = 0                        # entries past topk_length are ignored whatever they hold
    o2, l2, _ = orc.sparse_decode(q, sc.kv8.numpy(), ind.numpy(), sc.topk_length.numpy(), sc.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ---------------------------------------------------------------- packed selected-KV path

def test_pack_by_hand():
    """Each record's bytes encode its slot, so every packed slot can be checked
    against a value written out here, without the oracle's gather."""
    pages = 3
    slot = np.arange(pages * 64)[:, None]
    kv8 = ((slot * 7 + np.arange(656)[None, :]) % 251).astype(np.uint8).reshape(pages, 64, 656)
    rng = np.random.default_rng(21)
    ind = rng.integers(0, pages * 64, size=(1, 2, 70)).astype(np.int32)
    ind[0, 0, 3] = -1
    ind[0, 0, 10] = pages * 64                # outside the pool: masked, counted
    ind[0, 1, 66] = -7                        # past unit 1's prefix: ignored, not counted
    tl = np.array([[70, 65]], dtype=np.int32)
    packed, bad = orc.pack_selected(kv8, ind, tl)
    assert bad == 1
    assert packed.size == 2 * 2 * (64 * 656 + 8)
    records = packed[:2 * 128 * 656].reshape(2, 128, 656)
    masks = packed[2 * 128 * 656:].view(np.uint64).reshape(2, 2)
    for u in range(2):
        for t in range(128):
            valid = t < tl[0, u] and not (u == 0 and t in (3, 10))
            want = (int(ind[0, u, t]) * 7 + np.arange(656)) % 251 if valid else np.zeros(656)
            assert np.array_equal(records[u, t], want.astype(np.uint8)), (u, t)
    full = (1 << 64) - 1
    assert int(masks[0, 0]) == full & ~(1 << 3) & ~(1 << 10)
    assert int(masks[0, 1]) == 0x3F           # slots 64..69
    assert int(masks[1, 0]) == full and int(masks[1, 1]) == 0x1


def test_packed_workspace_size_matches_page():
    facts = json.load(open(os.path.join(GOLDEN, "page_facts.json")))
    f = facts["packed_workspace_per_row_topk2048"]
    tiles, rec, total = orc.packed_layout(1, f["topk"])
    assert tiles == 32 and round(rec / 2 ** 20, 3) == f["value_mib"]
    assert round(total / 2 ** 20, 3) == f["value_mib"]          # the masks add 256 B per row


def test_packed_decode_equals_native_sparse():
    sc = wl.sparse_case(2, 2, 8, topk=130, pages_per_req=4, topk_lengths=[[130, 77], [1, 0]], seed=22)
    ind = sc.indices.clone()
    ind[0, 0, ::9] = -1
    ind[0, 1, 5] = sc.kv8.shape[0] * 64 + 3
    q = f64(sc.q)
    o1, l1, bad1 = orc.sparse_decode(q, sc.kv8.numpy(), ind.numpy(), sc.topk_length.numpy(), sc.scale)
    packed, bad2 = orc.pack_selected(sc.kv8.numpy(), ind.numpy(), sc.topk_length.numpy())
    o2, l2 = orc.packed_decode(q, packed, 130, sc.topk_length.numpy(), sc.scale)
    assert bad1 == bad2 == 1
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    assert np.isneginf(l2[1, 1]).all() and not o2[1, 1].any()


def test_packed_mask_bit_controls_the_slot():
    """Clearing one mask bit equals masking that entry in the native selection."""
    sc = wl.sparse_case(1, 1, 4, topk=64, pages_per_req=2, topk_lengths=[[64]], seed=23)
    q = f64(sc.q)
    packed, _ = orc.pack_selected(sc.kv8.numpy(), sc.indices.numpy(), None)
    _, rec, _ = orc.packed_layout(1, 64)
    m = packed[rec:].view(np.uint64)
    m[0] &= ~np.uint64(1 << 17)
    o1, l1 = orc.packed_decode(q, packed, 64, None, sc.scale)
    ind = sc.indices.clone()
    ind[0, 0, 17] = -1
    o2, l2, _ = orc.sparse_decode(q, sc.kv8.numpy(), ind.numpy(), None, sc.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ---------------------------------------------------------------- several latent KV heads, fp16 inputs

def sdpa_grouped_reference(case, b):
    """torch fp64 SDPA with the KV heads expanded to the query heads by repeat_interleave
    (enable_gqa-style grouping done by hand), keys gathered with torch indexing."""
    L = int(case.cache_seqlens[b])
    h_kv = case.kv.shape[2]
    flat = case.kv.double().reshape(-1, h_kv, 576)             # [slots, h_kv, 576]
    j = torch.arange(L)
    slot = case.block_table[b].long()[j // 64] * 64 + (j % 64)
    K = flat[slot].permute(1, 0, 2)                             # [h_kv, L, 576]
    s_q, h_q = case.s_q, case.h_q
    K = K.repeat_interleave(h_q // h_kv, dim=0)                 # [h_q, L, 576]
    q = case.q[b].double().permute(1, 0, 2)                     # [h_q, s_q, 576]
    tok = torch.arange(s_q)
    allowed = (j[None, :] <= (L - s_q + tok[:, None])) if case.causal else torch.ones(s_q, L, dtype=torch.bool)
    bias = torch.zeros(s_q, L, dtype=torch.float64).masked_fill(~allowed, float("-inf"))
    out = torch.nn.functional.scaled_dot_product_attention(q, K, K[..., :512], attn_mask=bias, scale=case.scale)
    lse = torch.logsumexp(q @ K.transpose(1, 2) * case.scale + bias, dim=-1)
    return out.permute(1, 0, 2).numpy(), lse.T.numpy()


@pytest.mark.parametrize("h_kv,h_q,s_q,causal", [(2, 8, 1, False), (4, 16, 2, True), (3, 6, 3, True)])
def test_grouped_kv_heads_match_torch_sdpa(h_kv, h_q, s_q, causal):
    case = wl.dense_case(2, s_q, h_q, 0, seqlens=[70, 150], causal=causal, h_kv=h_kv, seed=h_kv * 10 + s_q)
    assert case.kv.shape[2] == h_kv
    out, lse = orc.dense_decode(f64(case.q), f64(case.kv), case.block_table.numpy(), case.cache_seqlens.numpy(),
                                case.causal, case.scale)
    for b in range(2):
        ro, rl = sdpa_grouped_reference(case, b)
        assert np.abs(out[b] - ro).max() < TOL and np.abs(lse[b] - rl).max() < TOL


def test_identical_kv_heads_reduce_to_one_head():
    one = wl.dense_case(1, 2, 8, 0, seqlens=[200], causal=True, seed=77)
    kv2 = torch.stack([one.kv, one.kv], dim=2)                 # [pages, 64, 2, 576], both heads equal
    o1, l1 = orc.dense_decode(f64(one.q), f64(one.kv), one.block_table.numpy(), one.cache_seqlens.numpy(), True,
                              one.scale)
    o2, l2 = orc.dense_decode(f64(one.q), f64(kv2), one.block_table.numpy(), one.cache_seqlens.numpy(), True,
                              one.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_swapping_kv_heads_swaps_head_groups():
    case = wl.dense_case(1, 1, 8, 0, seqlens=[130], h_kv=2, seed=78)
    q = f64(case.q)
    o, l = orc.dense_decode(q, f64(case.kv), case.block_table.numpy(), case.cache_seqlens.numpy(), False, case.scale)
    q_sw = np.concatenate([q[:, :, 4:], q[:, :, :4]], axis=2)
    o_sw, l_sw = orc.dense_decode(q_sw, f64(case.kv.flip(2)), case.block_table.numpy(), case.cache_seqlens.numpy(),
                                  False, case.scale)
    assert np.array_equal(o_sw[:, :, 4:], o[:, :, :4]) and np.array_equal(o_sw[:, :, :4], o[:, :, 4:])
    assert np.array_equal(l_sw[:, :, 4:], l[:, :, :4])


def test_fp16_case_holds_exact_fp16_values():
    case = wl.dense_case(1, 1, 4, 0, seqlens=[64], dtype=torch.float16, seed=79)
    assert case.q.dtype == torch.float16 and case.kv.dtype == torch.float16
    out, lse = orc.dense_decode(f64(case.q), f64(case.kv), case.block_table.numpy(), case.cache_seqlens.numpy(),
                                False, case.scale)
    ro, rl = sdpa_dense_reference(case, 0)
    assert np.abs(out[0] - ro).max() < TOL and np.abs(lse[0] - rl).max() < TOL


# ---------------------------------------------------------------- dense decode over FP8 records

@pytest.mark.parametrize("s_q,causal", [(1, False), (2, True), (3, True)])
def test_dense_fp8_equals_dense_on_decoded_records(s_q, causal):
    """Same keys, same order: decoding every record first and running the bf16-path oracle gives
    the same fp64 result; the records are decoded by torch's own fp8/bf16 conversions here."""
    case = wl.dense_fp8_case(2, s_q, 8, 0, seqlens=[70, 200], causal=causal, seed=80 + s_q)
    kv = torch_decode_records(case.kv8, torch.arange(case.kv8.shape[0] * 64)).reshape(-1, 64, 576)
    o1, l1 = orc.dense_fp8_decode(f64(case.q), case.kv8.numpy(), case.block_table.numpy(),
                                  case.cache_seqlens.numpy(), causal, case.scale)
    o2, l2 = orc.dense_decode(f64(case.q), kv.numpy(), case.block_table.numpy(), case.cache_seqlens.numpy(), causal,
                              case.scale)
    assert np.abs(o1 - o2).max() < TOL and np.abs(l1 - l2).max() < TOL


def test_dense_fp8_equals_sparse_over_every_slot():
    case = wl.dense_fp8_case(2, 1, 4, 0, seqlens=[130, 64], seed=84)
    bt = case.block_table.numpy()
    L = case.cache_seqlens.numpy()
    ind = np.full((2, 1, 192), -1, dtype=np.int64)
    for b in range(2):
        j = np.arange(L[b])
        ind[b, 0, :L[b]] = bt[b, j // 64] * 64 + j % 64
    o1, l1 = orc.dense_fp8_decode(f64(case.q), case.kv8.numpy(), bt, L, False, case.scale)
    o2, l2, bad = orc.sparse_decode(f64(case.q), case.kv8.numpy(), ind, None, case.scale)
    assert bad == 0 and np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ---------------------------------------------------------------- out-of-pool block-table entries

@pytest.mark.parametrize("bad_entry", [-3, 10 ** 6])
def test_dense_out_of_pool_page_masks_its_keys(bad_entry):
    """A block-table entry outside [0, num_pages) removes that logical page's
    64 keys: torch SDPA over the remaining keys (gathered by torch indexing,
    the page dropped by position) gives the same rows; other requests are
    untouched."""
    case = wl.dense_case(2, 2, 8, 0, seqlens=[300, 150], causal=True, seed=61)
    bt = case.block_table.clone()
    bt[0, 2] = bad_entry                              # keys 128..191 of request 0
    out, lse = orc.dense_decode(f64(case.q), f64(case.kv), bt.numpy(), case.cache_seqlens.numpy(), True,
                                case.scale)
    L = 300
    j = torch.arange(L)
    keep = (j // 64) != 2
    slot = case.block_table[0].long()[j // 64] * 64 + (j % 64)
    K = case.kv.double().reshape(-1, 576)[slot[keep]]
    q = case.q[0].double().reshape(16, 576)
    tok = torch.arange(16) // 8
    allowed = j[keep][None, :] <= (L - 2 + tok[:, None])
    bias = torch.zeros(16, int(keep.sum()), dtype=torch.float64).masked_fill(~allowed, float("-inf"))
    ro = torch.nn.functional.scaled_dot_product_attention(q[None], K[None], K[None, :, :512], attn_mask=bias[None],
                                                          scale=case.scale)[0]
    rl = torch.logsumexp(q @ K.T * case.scale + bias, dim=-1)
    assert np.abs(out[0].reshape(16, 512) - ro.numpy()).max() < TOL
    assert np.abs(lse[0].reshape(16) - rl.numpy()).max() < TOL
    good_o, good_l = orc.dense_decode(f64(case.q), f64(case.kv), case.block_table.numpy(),
                                      case.cache_seqlens.numpy(), True, case.scale)
    assert np.array_equal(out[1], good_o[1]) and np.array_equal(lse[1], good_l[1])


def test_dense_fp8_out_of_pool_page_equals_sparse_with_those_slots_masked():
    case = wl.dense_fp8_case(2, 1, 4, 0, seqlens=[200, 64], seed=85)
    bt = case.block_table.numpy().copy()
    L = case.cache_seqlens.numpy()
    ind = np.full((2, 1, 256), -1, dtype=np.int64)
    for b in range(2):
        j = np.arange(L[b])
        ind[b, 0, :L[b]] = bt[b, j // 64] * 64 + j % 64
    bt[0, 1] = case.kv8.shape[0]                      # keys 64..127 of request 0: one past the pool
    ind[0, 0, 64:128] = -1
    o1, l1 = orc.dense_fp8_decode(f64(case.q), case.kv8.numpy(), bt, L, False, case.scale)
    o2, l2, bad = orc.sparse_decode(f64(case.q), case.kv8.numpy(), ind, None, case.scale)
    assert bad == 0 and np.array_equal(o1, o2) and np.array_equal(l1, l2)
