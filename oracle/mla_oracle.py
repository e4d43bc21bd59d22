"""CPU fp64 oracle for MLA decode over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only
the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code, table or constant generator
with the CUDA path.

What is computed, and where the pages define it
-----------------------------------------------
Dense decode (FlashMLA PR #183, "Add SM80 (Ampere/A100) dense MLA decode
kernel", sections *Design* and *Test plan*): every query token carries h_q
heads that all attend to ONE latent KV head.  A key row has 576 entries
(512 "NoPE" + 64 "RoPE"), the score is the dot product over all 576, and the
value is the first 512 entries of the same row (each of the four warpgroups
in the page's design owns HEAD_DIM_V/4 = 128 value columns, so d_v = 512).
The cache is paged, 64 tokens per page, and a per-request block table maps a
logical page to a physical page.  Multi-token queries use a causal mask.
The output is softmax(Q K^T * scale) V per row plus the row's log-sum-exp.

Split-KV (same page, *Test plan*, which checks split-K through the combine
kernel; *Modifications outside csrc/sm80/*, which lists that kernel): the keys of one request can be cut
into splits, each producing a partial output and an LSE, which the combine
step merges.  ``split_partials`` / ``combine_partials`` restate that.

Sparse FP8 decode (FlashMLA PR #200, "[SM90] Add packed selected-KV sparse
decode", sections *Motivation* and *SM90 packing kernel*): each query token
selects up to top-k PHYSICAL slot indices into a pool of 656-byte records
(512 B of FP8 E4M3 NoPE values, 16 B holding four fp32 scales, 128 B holding
64 bf16 RoPE values); an index is split into a page and an in-page position;
``topk_length`` gives the valid prefix of the selection.  Attention then
runs over the dequantised records exactly as in the dense case.

Readings taken where the pages are silent (each is listed in the design doc):
  * LSE is the natural log of the sum of exp(scaled score).
  * Causal alignment is bottom-right: query token i of s_q sees keys
    j <= L - s_q + i (cache_seqlens already count the new tokens).
  * A row with no valid key gets out = 0 and lse = -inf.
  * Sparse: index -1 is masked anywhere; entries at or past topk_length are
    masked; a duplicated index counts as two keys; an index outside
    [0, num_pages*64) is masked and reported.
  * Dense: a block-table entry outside [0, num_pages) masks the 64 keys of
    that logical page (the same reading as an out-of-pool sparse index).
  * Record bytes are contiguous in the order the page lists them:
    [0,512) E4M3 codes, [512,528) four little-endian fp32 scales,
    [528,656) 64 little-endian bf16.  Element d < 512 uses scale d // 128.
  * E4M3 is the "fn" variant: bias 7, no infinities, S.1111.111 is NaN.

All floating point here is float64 except ``unpack_records``, whose result
is defined in fp32 (one IEEE round-to-nearest-even multiply per element).
"""

from __future__ import annotations

import numpy as np

PAGE_SIZE = 64          # tokens per KV page (PR #183, *How the occupancy work went*)
D_QK = 576              # 512 NoPE + 64 RoPE (PR #183 *Design*; PR #200 record layout)
D_V = 512               # value = first 512 entries of the latent row
RECORD_BYTES = 656      # PR #200 *SM90 packing kernel*: 512 + 16 + 128
NOPE_BYTES = 512
SCALE_OFF = 512
ROPE_OFF = 528
GROUP = 128             # one fp32 scale per 128 NoPE elements (four scales)


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------

def e4m3fn_to_f64(codes) -> np.ndarray:
    """Decode FP8 E4M3 ("fn": bias 7, no inf, 0x7F/0xFF = NaN) to float64.

    Bit layout: s eeee mmm.  e == 0 is subnormal: (-1)^s * 2^-6 * m/8.
    Otherwise (-1)^s * 2^(e-7) * (1 + m/8).  e == 15 and m == 7 is NaN.
    PR #200 (*SM90 packing kernel*) stores the NoPE part of its 656-byte
    record in this format.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    sign = np.where(s == 1, -1.0, 1.0)
    sub = sign * np.ldexp(m.astype(np.float64) / 8.0, -6)
    nrm = sign * np.ldexp(1.0 + m.astype(np.float64) / 8.0, (e - 7).astype(np.int64))
    out = np.where(e == 0, sub, nrm)
    out = np.where((e == 15) & (m == 7), np.nan, out)
    return out


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64: the bf16 is the top half of an fp32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _le_f32(byte_block: np.ndarray) -> np.ndarray:
    """Little-endian fp32 values from a [..., 4k] uint8 block."""
    b = np.ascontiguousarray(byte_block, dtype=np.uint8)
    return b.view("<f4")


def _le_u16(byte_block: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(byte_block, dtype=np.uint8)
    return b.view("<u2")


# --------------------------------------------------------------------------
# Key gathering
# --------------------------------------------------------------------------

def dense_keys(kv: np.ndarray, block_table: np.ndarray, b: int, L: int):
    """Latent rows of request b in logical order 0..L-1, read through the block table.

    Logical token j lives in physical page block_table[b][j // 64] at slot
    j % 64 (PR #183: 64-token pages; the block table maps logical to
    physical pages).  Returns (rows [L, 576], present [L]): a token whose
    page entry lies outside [0, num_pages) is absent (zero row, masked).
    """
    rows = np.zeros((L, D_QK), dtype=np.float64)
    present = np.zeros(L, dtype=bool)
    for j in range(L):
        page = int(block_table[b, j // PAGE_SIZE])
        if 0 <= page < kv.shape[0]:
            rows[j] = kv[page, j % PAGE_SIZE]
            present[j] = True
    return rows, present


def decode_record(rec: np.ndarray) -> np.ndarray:
    """One 656-byte record -> its 576 key values in float64 (exact).

    k[d]       = e4m3(rec[d]) * scale[d // 128]      for d < 512
    k[512 + e] = bf16(rope[e])                       for e < 64
    (PR #200 *SM90 packing kernel* lists the three parts in this order.)
    """
    rec = np.asarray(rec, dtype=np.uint8)
    assert rec.shape == (RECORD_BYTES,)
    nope = e4m3fn_to_f64(rec[:NOPE_BYTES])
    scales = _le_f32(rec[SCALE_OFF:ROPE_OFF]).astype(np.float64)
    rope = bf16_bits_to_f64(_le_u16(rec[ROPE_OFF:RECORD_BYTES]))
    k = np.empty(D_QK, dtype=np.float64)
    k[:NOPE_BYTES] = nope * np.repeat(scales, GROUP)     # element d uses scale d // 128
    k[NOPE_BYTES:] = rope
    return k


def slot_valid(idx: int, t: int, topk_len: int, num_slots: int) -> tuple[bool, bool]:
    """(is_key, is_bad_index) for selection entry t holding index idx."""
    if t >= topk_len or idx == -1:
        return False, False
    if idx < 0 or idx >= num_slots:
        return False, True
    return True, False


def sparse_keys(kv8: np.ndarray, idx_row: np.ndarray, topk_len: int):
    """Keys selected by one query token: list of decoded rows (duplicates kept).

    An index is a physical slot: page = idx // 64, in-page position idx % 64
    (PR #200 *Motivation* names this index-to-page translation as work the
    native kernel does).  Returns (rows[n, 576], bad_index_count).
    """
    num_pages = kv8.shape[0]
    rows = []
    bad = 0
    for t in range(idx_row.shape[0]):
        idx = int(idx_row[t])
        ok, is_bad = slot_valid(idx, t, topk_len, num_pages * PAGE_SIZE)
        bad += int(is_bad)
        if ok:
            rows.append(decode_record(kv8[idx // PAGE_SIZE, idx % PAGE_SIZE]))
    if rows:
        return np.stack(rows), bad
    return np.zeros((0, D_QK), dtype=np.float64), bad


# --------------------------------------------------------------------------
# Attention of a block of rows over a key set
# --------------------------------------------------------------------------

def attend(qrows: np.ndarray, keys: np.ndarray, scale: float, valid: np.ndarray | None = None):
    """softmax(q K^T * scale) V with V = K[:, :512]; returns (out[R, 512], lse[R]).

    ``valid`` is an optional boolean [R, n] mask.  A row with no valid key
    gets out = 0, lse = -inf.  LSE is ln(sum_j exp(s_j)).
    """
    R = qrows.shape[0]
    n = keys.shape[0]
    out = np.zeros((R, D_V), dtype=np.float64)
    lse = np.full(R, -np.inf, dtype=np.float64)
    if n == 0:
        return out, lse
    s = (qrows @ keys.T) * scale                      # [R, n] scaled scores
    if valid is None:
        valid = np.ones((R, n), dtype=bool)
    m = np.where(valid, s, -np.inf).max(axis=1)       # row max over valid keys
    has = np.isfinite(m)
    m_safe = np.where(has, m, 0.0)
    # masked keys get weight exactly 0, so their values never reach the sums
    w = np.where(valid, np.exp(s - m_safe[:, None]), 0.0)
    z = w.sum(axis=1)
    pv = w @ keys[:, :D_V]                            # V = first 512 entries
    out[has] = pv[has] / z[has, None]
    lse[has] = m[has] + np.log(z[has])
    return out, lse


def causal_mask(s_q: int, h_q: int, L: int, causal: bool) -> np.ndarray:
    """[s_q*h_q, L] validity: row r is query token i = r // h_q; with causal,
    it sees keys j <= L - s_q + i (bottom-right alignment)."""
    R = s_q * h_q
    j = np.arange(L)[None, :]
    i = (np.arange(R) // h_q)[:, None]
    if not causal:
        return np.ones((R, L), dtype=bool)
    return j <= (L - s_q + i)


# --------------------------------------------------------------------------
# Dense and sparse decode
# --------------------------------------------------------------------------

def dense_decode(q, kv, block_table, cache_seqlens, causal, scale, batches=None):
    """Dense MLA paged decode.

    q: [B, s_q, h_q, 576]; kv: [num_pages, 64, 576], or [num_pages, 64, h_kv,
    576] for h_kv latent KV heads (PR #183 *Test plan* sweeps hk = 1..4); any
    real dtype, used as float64.  Query head h reads KV head h // (h_q // h_kv)
    (the pages do not spell the grouping out: consecutive query heads share a
    KV head, the usual grouped-query reading).  block_table: [B, max_pages]
    int, cache_seqlens: [B] int.  Returns out [B, s_q, h_q, 512] and lse
    [B, s_q, h_q] in float64.  ``batches`` restricts the work to a subset of
    requests (others stay 0/-inf).
    """
    q = np.asarray(q, dtype=np.float64)
    kv = np.asarray(kv)          # gathered rows are widened to float64 one by one
    if kv.ndim == 3:
        kv = kv[:, :, None, :]
    B, s_q, h_q, _ = q.shape
    h_kv = kv.shape[2]
    assert h_q % h_kv == 0
    G = h_q // h_kv
    out = np.zeros((B, s_q, h_q, D_V), dtype=np.float64)
    lse = np.full((B, s_q, h_q), -np.inf, dtype=np.float64)
    for b in (range(B) if batches is None else batches):
        L = int(cache_seqlens[b])
        for g in range(h_kv):
            keys, present = dense_keys(kv[:, :, g, :], block_table, b, L)
            heads = slice(g * G, (g + 1) * G)
            qrows = q[b][:, heads, :].reshape(s_q * G, D_QK)
            o, l = attend(qrows, keys, scale, causal_mask(s_q, G, L, causal) & present[None, :])
            out[b][:, heads] = o.reshape(s_q, G, D_V)
            lse[b][:, heads] = l.reshape(s_q, G)
    return out, lse


def dense_fp8_decode(q, kv8, block_table, cache_seqlens, causal, scale, batches=None):
    """Dense decode over a paged cache of 656-byte FP8 records.

    PR #183 (*Limitations / future work*) lists an FP8 KV cache as what the
    SM80 dense kernel lacks, without a format; the only FP8 layout the pages
    define is PR #200's record (*SM90 packing kernel*), so that is the reading
    taken: kv8 [num_pages, 64, 656], token j of request b is record j % 64 of
    page block_table[b][j // 64], its key is ``decode_record`` of it, and the
    attention (all keys, causal alignment, LSE) is that of ``dense_decode``.
    Returns out [B, s_q, h_q, 512] and lse [B, s_q, h_q] in float64.
    """
    q = np.asarray(q, dtype=np.float64)
    kv8 = np.asarray(kv8, dtype=np.uint8)
    B, s_q, h_q, _ = q.shape
    out = np.zeros((B, s_q, h_q, D_V), dtype=np.float64)
    lse = np.full((B, s_q, h_q), -np.inf, dtype=np.float64)
    for b in (range(B) if batches is None else batches):
        L = int(cache_seqlens[b])
        keys = np.zeros((L, D_QK), dtype=np.float64)
        present = np.zeros(L, dtype=bool)          # out-of-pool page entries mask their keys
        for j in range(L):
            page = int(block_table[b, j // PAGE_SIZE])
            if 0 <= page < kv8.shape[0]:
                keys[j] = decode_record(kv8[page, j % PAGE_SIZE])
                present[j] = True
        qrows = q[b].reshape(s_q * h_q, D_QK)
        o, l = attend(qrows, keys, scale, causal_mask(s_q, h_q, L, causal) & present[None, :])
        out[b] = o.reshape(s_q, h_q, D_V)
        lse[b] = l.reshape(s_q, h_q)
    return out, lse


def sparse_decode(q, kv8, indices, topk_length, scale, batches=None):
    """Sparse FP8 MLA decode over selected 656-byte records.

    q: [B, s_q, h_q, 576]; kv8: uint8 [num_pages, 64, 656];
    indices: [B, s_q, topk] int; topk_length: [B, s_q] int or None (= topk).
    Returns (out [B, s_q, h_q, 512], lse [B, s_q, h_q], bad_index_count).
    """
    q = np.asarray(q, dtype=np.float64)
    kv8 = np.asarray(kv8, dtype=np.uint8)
    B, s_q, h_q, _ = q.shape
    topk = indices.shape[2]
    out = np.zeros((B, s_q, h_q, D_V), dtype=np.float64)
    lse = np.full((B, s_q, h_q), -np.inf, dtype=np.float64)
    bad_total = 0
    for b in (range(B) if batches is None else batches):
        for i in range(s_q):
            tl = topk if topk_length is None else int(topk_length[b, i])
            keys, bad = sparse_keys(kv8, indices[b, i], tl)
            bad_total += bad
            o, l = attend(q[b, i], keys, scale)
            out[b, i] = o
            lse[b, i] = l
    return out, lse, bad_total


# --------------------------------------------------------------------------
# Packed selected-KV path
# --------------------------------------------------------------------------

def packed_layout(n_units: int, topk: int):
    """(tiles, records_bytes, total_bytes) of the packed workspace.

    PR #200 *SM90 packing kernel*: an opaque workspace of 64-token tiles.
    This library fixes it as uint8 [n_units, tiles, 64, 656] records, then
    uint64 [n_units, tiles] valid masks, tiles = ceil(topk / 64).
    """
    tiles = -(-topk // PAGE_SIZE)
    records = n_units * tiles * PAGE_SIZE * RECORD_BYTES
    return tiles, records, records + n_units * tiles * 8


def pack_selected(kv8, indices, topk_length):
    """Byte-for-byte copy of every selected record into the packed layout.

    PR #200 *SM90 packing kernel*: each selected record is copied unchanged;
    slots past the valid prefix (topk_length) are zero-filled.  Slots the
    native selection masks (-1, or an index outside the pool) are zero-filled
    and left out of the tile's valid mask too.
    Returns (packed uint8 1-D, bad_index_count).
    """
    kv8 = np.asarray(kv8, dtype=np.uint8)
    B, s_q, topk = indices.shape
    n_units = B * s_q
    num_slots = kv8.shape[0] * PAGE_SIZE
    tiles, rec_bytes, total = packed_layout(n_units, topk)
    packed = np.zeros(total, dtype=np.uint8)
    records = packed[:rec_bytes].reshape(n_units, tiles * PAGE_SIZE, RECORD_BYTES)
    masks = np.zeros((n_units, tiles), dtype=np.uint64)
    bad = 0
    for b in range(B):
        for i in range(s_q):
            u = b * s_q + i
            tl = topk if topk_length is None else int(topk_length[b, i])
            for t in range(topk):
                idx = int(indices[b, i, t])
                ok, is_bad = slot_valid(idx, t, tl, num_slots)
                bad += int(is_bad)
                if ok:
                    records[u, t] = kv8[idx // PAGE_SIZE, idx % PAGE_SIZE]
                    masks[u, t // PAGE_SIZE] |= np.uint64(1) << np.uint64(t % PAGE_SIZE)
    packed[rec_bytes:] = masks.reshape(-1).view(np.uint8)
    return packed, bad


def packed_decode(q, packed, topk, topk_length, scale):
    """Sparse decode over a packed workspace (PR #200 *Packed attention
    specialization*): slot t of unit u is a key iff t < topk_length and its
    bit in the tile mask is set; its record sits at a fixed position.
    Returns (out [B, s_q, h_q, 512], lse [B, s_q, h_q])."""
    q = np.asarray(q, dtype=np.float64)
    B, s_q, h_q, _ = q.shape
    n_units = B * s_q
    tiles, rec_bytes, total = packed_layout(n_units, topk)
    packed = np.asarray(packed, dtype=np.uint8)
    assert packed.shape == (total,)
    records = packed[:rec_bytes].reshape(n_units, tiles * PAGE_SIZE, RECORD_BYTES)
    masks = packed[rec_bytes:].view(np.uint64).reshape(n_units, tiles)
    out = np.zeros((B, s_q, h_q, D_V), dtype=np.float64)
    lse = np.full((B, s_q, h_q), -np.inf, dtype=np.float64)
    for b in range(B):
        for i in range(s_q):
            u = b * s_q + i
            tl = min(topk, topk if topk_length is None else int(topk_length[b, i]))
            rows = [decode_record(records[u, t]) for t in range(max(tl, 0))
                    if (int(masks[u, t // PAGE_SIZE]) >> (t % PAGE_SIZE)) & 1]
            keys = np.stack(rows) if rows else np.zeros((0, D_QK), dtype=np.float64)
            out[b, i], lse[b, i] = attend(q[b, i], keys, scale)
    return out, lse


# --------------------------------------------------------------------------
# Split-KV partials and the combine step
# --------------------------------------------------------------------------

def split_partials(qrows, keys, scale, cuts, valid=None):
    """Per-split (O_s, lse_s) for key ranges [cuts[k], cuts[k+1]).

    Each split is an independent softmax over its own keys (PR #183 *Test
    plan* exercises split-K through the combine kernel).  Empty splits give O = 0,
    lse = -inf.
    """
    parts = []
    for a, z in zip(cuts[:-1], cuts[1:]):
        vs = None if valid is None else valid[:, a:z]
        parts.append(attend(qrows, keys[a:z], scale, vs))
    return parts


def combine_partials(parts):
    """Merge split partials: L = ln sum_s exp(lse_s), out = sum_s exp(lse_s - L) O_s.

    A split with lse = -inf has weight 0; if every split is empty the row is
    out = 0, lse = -inf.
    """
    O = np.stack([p[0] for p in parts])          # [S, R, 512]
    LS = np.stack([p[1] for p in parts])         # [S, R]
    R = O.shape[1]
    out = np.zeros((R, D_V), dtype=np.float64)
    lse = np.full(R, -np.inf, dtype=np.float64)
    for r in range(R):
        col = LS[:, r]
        fin = np.isfinite(col)
        if not fin.any():
            continue
        m = col[fin].max()
        w = np.where(fin, np.exp(np.where(fin, col, m) - m), 0.0)
        z = w.sum()
        out[r] = (w[:, None] * O[:, r]).sum(axis=0) / z
        lse[r] = m + np.log(z)
    return out, lse


# --------------------------------------------------------------------------
# Bit-exact record gather + unpack (fp32)
# --------------------------------------------------------------------------

def unpack_records(kv8, idx_flat):
    """Gather records by physical slot index and unpack them to fp32 rows.

    k[d] = fp32(e4m3(code_d)) * fp32(scale[d // 128]) as ONE fp32
    round-to-nearest-even multiply (d < 512); k[512+e] = fp32(bf16 rope[e]).
    Index -1 or an index outside the pool gives a zero row; the second
    return value counts out-of-pool indices.
    """
    kv8 = np.asarray(kv8, dtype=np.uint8)
    num_slots = kv8.shape[0] * PAGE_SIZE
    idx_flat = np.asarray(idx_flat).reshape(-1)
    out = np.zeros((idx_flat.shape[0], D_QK), dtype=np.float32)
    bad = 0
    for n, idx in enumerate(idx_flat.tolist()):
        if idx == -1:
            continue
        if idx < 0 or idx >= num_slots:
            bad += 1
            continue
        rec = kv8[idx // PAGE_SIZE, idx % PAGE_SIZE]
        nope = e4m3fn_to_f64(rec[:NOPE_BYTES]).astype(np.float32)   # exact
        scales = _le_f32(rec[SCALE_OFF:ROPE_OFF]).astype(np.float32)
        for g in range(NOPE_BYTES // GROUP):
            seg = slice(g * GROUP, (g + 1) * GROUP)
            out[n, seg] = nope[seg] * scales[g]                      # fp32 RNE
        out[n, NOPE_BYTES:] = bf16_bits_to_f64(_le_u16(rec[ROPE_OFF:])).astype(np.float32)
    return out, bad
