"""kvq oracle: a plain, slow CPU definition of decode attention over an
asymmetric INT2/INT4 group-quantized KV cache (numpy, fp64).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import this package. The CUDA
library neither imports nor calls it, and it imports nothing from the CUDA
library: the two share no code, tables or constants.

Sources -- three web pages about the FOSCAR preprint (arXiv 2611.09722):

  [ABS]  "FOSCAR: Accelerating Decode Attention over 2- and 4-Bit KV Caches
         through Affine Folding" (papers.pytorch.kr), the abstract.
  [NEWS] "FOSCAR boosts LLM decode attention 3.4x using 2-bit KV caches"
         (grafy.ai), section "What is FOSCAR and how does it work?".
  [SUM]  rag-lover.com summary of arXiv 2611.09722, sections
         "使える条件" (conditions of use), "限界と未検証の範囲" (limits) and
         "解説" (commentary).

What the pages fix: each cached value is a 2- or 4-bit integer; a group of
values shares one scale s and one offset z (asymmetric quantization) and K and
V each use either token-wise or channel-wise groups ([SUM] 使える条件; [NEWS]).
Group size 128 appears in [SUM] 使える条件.  The folded form is exactly equal
to dequantize-then-attend ([ABS]; [SUM] 解説).

Readings taken where the pages are silent (the reconstruction formula itself is
lost in the [NEWS] extraction):

  * reconstruction: x_hat = s * q + z with q unsigned in [0, 2^b - 1];
  * quantizer: z = fp16 rounded toward -inf of the group minimum,
    s = fp16 rounded toward +inf of fp32((max - z) / (2^b - 1)),
    q = clamp(rint_half_even(fp32(fp32(x - z) / s)), 0, 2^b - 1), every step
    an IEEE fp32 operation (no fused multiply-add); a group whose max equals z
    gets s = 0 and q = 0 (x_hat = z);
  * groups of G elements (G = 128 by default; [SUM] 使える条件 names 128,
    [SUM] 限界と未検証の範囲 says results depend on the group size):
    token-wise = G consecutive channels of one token of one KV head (G divides
    the head dim D); channel-wise = G consecutive tokens of one channel of one
    KV head, aligned to token 0 (G divides the 128-token block); a block's
    tokens at or past the sequence length are excluded from min/max and get
    code 0 (token-wise: s = z = 0 as well; a channel-wise group with no valid
    token: s = z = 0);
  * GQA: query head h reads KV head h // (Hq / Hkv);
  * scores S_l = sm_scale * q . x_hat_K[l], sm_scale = 1/sqrt(D) by default;
    lse = natural-log sum of exp(S_l); an empty sequence gives out = 0,
    lse = -inf;
  * packed layout: see ``pack_rows`` / ``page_of``.
"""
from __future__ import annotations

import math

import numpy as np

BLOCK_TOKENS = 128  # tokens per block (= page); also the channel-wise group
HEAD_DIM = 128  # default head dim; 64 and 256 are also covered
GROUP = 128     # default group size; 32 and 64 are also covered
TOKENWISE = 0
CHANNELWISE = 1
K_CACHE = 0
V_CACHE = 1


class OracleError(ValueError):
    """Raised for inputs the quantizer rejects (non-finite values, fp16 overflow)."""


# ---------------------------------------------------------------------------
# fp16 directed rounding and the bf16 query format
# ---------------------------------------------------------------------------

def fp16_round_down(x32):
    """fp32 -> fp16 rounded toward -inf (elementwise, returns np.float16)."""
    x32 = np.asarray(x32, dtype=np.float32)
    with np.errstate(over="ignore"):
        h = x32.astype(np.float16)  # round to nearest even (overflow -> inf)
        fix = h.astype(np.float32) > x32
        return np.where(fix, np.nextafter(h, np.float16(-np.inf)), h).astype(np.float16)


def fp16_round_up(x32):
    """fp32 -> fp16 rounded toward +inf (elementwise, returns np.float16)."""
    x32 = np.asarray(x32, dtype=np.float32)
    with np.errstate(over="ignore"):
        h = x32.astype(np.float16)
        fix = h.astype(np.float32) < x32
        return np.where(fix, np.nextafter(h, np.float16(np.inf)), h).astype(np.float16)


def bf16_bits_to_f64(bits):
    """bf16 bit patterns (uint16 array) -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# Quantization of one group  ([SUM] 使える条件: asymmetric, shared s and z)
# ---------------------------------------------------------------------------

def quantize_groups(X, bits):
    """Quantize each row of X (fp32 [g, n]) as one group.

    Returns (codes uint8 [g, n], s fp16 [g], z fp16 [g]); the reconstruction
    is x_hat = s * code + z.
    """
    X = np.asarray(X, dtype=np.float32)
    g, n = X.shape
    if n == 0:
        return np.zeros((g, 0), np.uint8), np.zeros(g, np.float16), np.zeros(g, np.float16)
    if not np.all(np.isfinite(X)):
        raise OracleError("non-finite value in a quantization group")
    qmax = (1 << bits) - 1
    lo = X.min(axis=1)
    hi = X.max(axis=1)
    z = fp16_round_down(lo)
    if not np.all(np.isfinite(z)):
        raise OracleError("group offset overflows fp16")
    rng = (hi - z.astype(np.float32)).astype(np.float32)           # fp32 subtract
    degenerate = rng == np.float32(0)
    s = fp16_round_up((rng / np.float32(qmax)).astype(np.float32))  # fp32 divide, round up
    if not np.all(np.isfinite(s)):
        raise OracleError("group scale overflows fp16")
    s = np.where(degenerate, np.float16(0), s).astype(np.float16)
    diff = (X - z.astype(np.float32)[:, None]).astype(np.float32)  # fp32 subtract
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (diff / s.astype(np.float32)[:, None]).astype(np.float32)  # fp32 divide
    q = np.clip(np.rint(t), 0, qmax)
    q = np.where(degenerate[:, None], 0, q).astype(np.uint8)
    return q, s, z


def quantize_group(xg, bits):
    """One group: (codes uint8 [n], s np.float16, z np.float16)."""
    q, s, z = quantize_groups(np.asarray(xg, np.float32)[None, :], bits)
    return q[0], s[0], z[0]


def dequantize_value(code, s, z):
    """x_hat = s * q + z in fp64 (exact: s, z are fp16 and q has <= 4 bits)."""
    return np.float64(s) * np.asarray(code, np.float64) + np.float64(z)


# ---------------------------------------------------------------------------
# One sequence of one KV head  -> logical per-block codes and s/z
# ---------------------------------------------------------------------------

def num_blocks(n_tokens):
    return (int(n_tokens) + BLOCK_TOKENS - 1) // BLOCK_TOKENS


def check_geometry(head_dim, group):
    if head_dim not in (64, 128, 256) or group not in (32, 64, 128) or group > head_dim:
        raise OracleError("head_dim must be 64, 128 or 256 and the group 32, 64 or 128 (at most head_dim)")


def sz_per_block(head_dim, group):
    """s (or z) values per 128-token block of one KV head: 128 * D / G."""
    return BLOCK_TOKENS * head_dim // group


def quantize_sequence(x_seq, bits, scheme, group=GROUP):
    """Quantize the valid tokens of one (sequence, KV head).

    x_seq: fp32 [n, D] holding exactly the valid tokens.
    Returns codes uint8 [nblk, 128 tokens, D channels] and s, z fp16
    [nblk, 128 * D / G]: token-wise, entry t * (D / G) + g belongs to channels
    [g G, (g + 1) G) of block token t; channel-wise, entry k * D + c belongs
    to channel c over block tokens [k G, (k + 1) G).  (G = D = 128: one entry
    per token, resp. per channel.)
    """
    x_seq = np.asarray(x_seq, dtype=np.float32)
    n, d = x_seq.shape
    check_geometry(d, group)
    nblk = num_blocks(n)
    codes = np.zeros((nblk, BLOCK_TOKENS, d), np.uint8)
    if scheme == TOKENWISE:  # one group = G consecutive channels of one token
        gpt = d // group
        ct, st, zt = quantize_groups(x_seq.reshape(n * gpt, group), bits)
        pad = nblk * BLOCK_TOKENS - n
        codes[:] = np.concatenate([ct.reshape(n, d), np.zeros((pad, d), np.uint8)]).reshape(nblk, BLOCK_TOKENS, d)
        s = np.concatenate([st.reshape(n, gpt), np.zeros((pad, gpt), np.float16)]).reshape(nblk, BLOCK_TOKENS * gpt)
        z = np.concatenate([zt.reshape(n, gpt), np.zeros((pad, gpt), np.float16)]).reshape(nblk, BLOCK_TOKENS * gpt)
    elif scheme == CHANNELWISE:  # one group = one channel over G consecutive valid tokens
        gpb = BLOCK_TOKENS // group
        s = np.zeros((nblk, gpb, d), np.float16)
        z = np.zeros((nblk, gpb, d), np.float16)
        for j in range(nblk):
            for k in range(gpb):
                t0 = j * BLOCK_TOKENS + k * group
                nv = min(group, n - t0)
                if nv <= 0:
                    continue
                cc, sc, zc = quantize_groups(x_seq[t0:t0 + nv].T, bits)
                codes[j, k * group:k * group + nv] = cc.T
                s[j, k] = sc
                z[j, k] = zc
        s = s.reshape(nblk, gpb * d)
        z = z.reshape(nblk, gpb * d)
    else:
        raise OracleError("unknown scheme")
    return codes, s, z


# ---------------------------------------------------------------------------
# Packed block layout
# ---------------------------------------------------------------------------

def block_bytes(bits, head_dim=HEAD_DIM):
    """Bytes of one packed block: 128 tokens x D channels of b-bit codes."""
    return BLOCK_TOKENS * head_dim * bits // 8


def block_rows(codes_tc, which):
    """Logical rows of a block: K rows are tokens (channels along the row),
    V rows are channels (tokens along the row)."""
    return codes_tc if which == K_CACHE else codes_tc.T


def pack_rows(rows, bits):
    """Pack a [128 rows, 128 columns] code matrix.

    Within a row, column i sits at bits [b*(i mod 8/b), b*(i mod 8/b) + b) of
    row byte floor(i*b/8) (little-endian, low bits first).  The row bytes are
    cut into 16-byte chunks and the block is stored chunk-major:
    byte offset = (chunk * 128 + row) * 16 + byte_in_chunk.
    """
    rows = np.asarray(rows, dtype=np.uint8)
    nrows, ncols = rows.shape
    per_byte = 8 // bits
    row_bytes = ncols * bits // 8
    packed = np.zeros((nrows, row_bytes), np.uint8)
    for k in range(per_byte):  # column i = per_byte * byte + k
        packed |= (rows[:, k::per_byte] << (bits * k)).astype(np.uint8)
    nchunk = row_bytes // 16
    return packed.reshape(nrows, nchunk, 16).transpose(1, 0, 2).reshape(-1).copy()


def unpack_rows(blob, bits, nrows=BLOCK_TOKENS, ncols=HEAD_DIM):
    """Inverse of ``pack_rows``."""
    blob = np.asarray(blob, dtype=np.uint8)
    per_byte = 8 // bits
    row_bytes = ncols * bits // 8
    nchunk = row_bytes // 16
    packed = blob.reshape(nchunk, nrows, 16).transpose(1, 0, 2).reshape(nrows, row_bytes)
    mask = (1 << bits) - 1
    rows = np.zeros((nrows, ncols), np.uint8)
    for k in range(per_byte):
        rows[:, k::per_byte] = (packed >> (bits * k)) & mask
    return rows


def page_of(b, j, max_blocks, page_table):
    """Page holding block j of sequence b: page_table[b, j] when a page table
    is given, else b * max_blocks + j (contiguous cache)."""
    if page_table is None:
        return b * max_blocks + j
    return int(page_table[b, j])


# ---------------------------------------------------------------------------
# Whole cache
# ---------------------------------------------------------------------------

def pack_cache(x, seq_lens, bits, scheme, which, page_table=None, num_pages=None, group=GROUP):
    """Quantize and pack K or V for a batch.

    x: fp32 [B, Hkv, Lcap, D]; only tokens < seq_lens[b] are read.
    Cache arrays: codes uint8 [num_pages, Hkv, block_bytes], s and z fp16
    [num_pages, Hkv, 128 * D / G].  Pages not covered by a sequence stay zero.
    """
    x = np.asarray(x, dtype=np.float32)
    B, Hkv, Lcap, D = x.shape
    max_blocks = num_blocks(Lcap) if page_table is None else page_table.shape[1]
    if num_pages is None:
        num_pages = B * max_blocks if page_table is None else int(np.max(page_table)) + 1
    check_geometry(D, group)
    codes = np.zeros((num_pages, Hkv, block_bytes(bits, D)), np.uint8)
    s = np.zeros((num_pages, Hkv, sz_per_block(D, group)), np.float16)
    z = np.zeros((num_pages, Hkv, sz_per_block(D, group)), np.float16)
    for b in range(B):
        n = int(seq_lens[b])
        for h in range(Hkv):
            c, sb, zb = quantize_sequence(x[b, h, :n], bits, scheme, group)
            for j in range(c.shape[0]):
                p = page_of(b, j, max_blocks, page_table)
                codes[p, h] = pack_rows(block_rows(c[j], which), bits)
                s[p, h] = sb[j]
                z[p, h] = zb[j]
    return codes, s, z


def unpack_cache(codes, s, z, seq_lens, bits, which, Lcap, page_table=None):
    """Logical view of a packed cache.

    Returns codes uint8 [B, Hkv, Lcap, D] (token, channel) and s, z fp16
    [B, Hkv, nblk, 128 * D / G] per block, laid out as stored (see
    quantize_sequence).  D follows from the block size, G from the s arrays.
    """
    B = len(seq_lens)
    Hkv = codes.shape[1]
    D = codes.shape[2] * 8 // (BLOCK_TOKENS * bits)
    max_blocks = num_blocks(Lcap) if page_table is None else page_table.shape[1]
    nblk = num_blocks(Lcap)
    out_c = np.zeros((B, Hkv, nblk * BLOCK_TOKENS, D), np.uint8)
    out_s = np.zeros((B, Hkv, nblk, s.shape[2]), np.float16)
    out_z = np.zeros((B, Hkv, nblk, s.shape[2]), np.float16)
    for b in range(B):
        for j in range(num_blocks(seq_lens[b])):
            p = page_of(b, j, max_blocks, page_table)
            for h in range(Hkv):
                rows = unpack_rows(codes[p, h], bits, BLOCK_TOKENS if which == K_CACHE else D,
                                   D if which == K_CACHE else BLOCK_TOKENS)
                tc = rows if which == K_CACHE else rows.T
                out_c[b, h, j * BLOCK_TOKENS:(j + 1) * BLOCK_TOKENS] = tc
                out_s[b, h, j] = s[p, h]
                out_z[b, h, j] = z[p, h]
    return out_c[:, :, :Lcap], out_s, out_z


def expand_sz(s_blk, scheme, head_dim, nv):
    """Per-element view [Hkv, nv, D] of one block's s (or z) values
    [Hkv, 128 * D / G] for its first nv tokens."""
    s_blk = np.asarray(s_blk, np.float64)
    Hkv, m = s_blk.shape
    group = BLOCK_TOKENS * head_dim // m
    if scheme == TOKENWISE:   # [token][channel group]
        per = s_blk.reshape(Hkv, BLOCK_TOKENS, head_dim // group)
        return np.repeat(per, group, axis=2)[:, :nv]
    per = s_blk.reshape(Hkv, BLOCK_TOKENS // group, head_dim)  # [token group][channel]
    return np.repeat(per, group, axis=1)[:, :nv]


def dequantize(codes_tc, s, z, seq_lens, scheme):
    """x_hat fp64 [B, Hkv, Lcap, D] from logical codes and per-block s/z;
    tokens at or past seq_lens[b] are 0."""
    B, Hkv, Lcap, D = codes_tc.shape
    xh = np.zeros((B, Hkv, Lcap, D), np.float64)
    for b in range(B):
        n = int(seq_lens[b])
        for j in range(num_blocks(n)):
            l0, l1 = j * BLOCK_TOKENS, min(n, (j + 1) * BLOCK_TOKENS)
            c = codes_tc[b, :, l0:l1].astype(np.float64)           # [Hkv, nv, D]
            sv = expand_sz(s[b, :, j], scheme, D, l1 - l0)
            zv = expand_sz(z[b, :, j], scheme, D, l1 - l0)
            xh[b, :, l0:l1] = sv * c + zv
    return xh


# ---------------------------------------------------------------------------
# Decode attention, directly (the problem statement)
# ---------------------------------------------------------------------------

def attend(q, khat, vhat, seq_lens, sm_scale=None):
    """out[b,h] = softmax(S) @ vhat[b, h//G], S = sm_scale * khat[b, h//G] @ q[b,h].

    q: fp64 [B, Hq, D]; khat, vhat: fp64 [B, Hkv, Lcap, D].
    Returns out fp64 [B, Hq, D] and lse fp64 [B, Hq] (natural log).
    """
    q = np.asarray(q, np.float64)
    B, Hq, D = q.shape
    Hkv = khat.shape[1]
    G = Hq // Hkv
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.full((B, Hq), -np.inf, np.float64)
    for b in range(B):
        n = int(seq_lens[b])
        if n == 0:
            continue
        for h in range(Hq):
            kv = h // G
            S = sm_scale * (khat[b, kv, :n] @ q[b, h])
            m = S.max()
            e = np.exp(S - m)
            den = e.sum()
            out[b, h] = (e @ vhat[b, kv, :n]) / den
            lse[b, h] = m + math.log(den)
    return out, lse


# ---------------------------------------------------------------------------
# Affine-folded decode attention in exact arithmetic (check only)
# ---------------------------------------------------------------------------

def attend_folded(q, kc, ks, kz, vc, vs, vz, seq_lens, k_scheme, v_scheme, sm_scale=None):
    """The folded formulation on integer codes, fp64.

    QK^T contracts over channels ([SUM] 解説): token-wise K folds on the
    accumulator (scale the partial q.code of each channel group by its s,
    add z * sum(q) over the group); channel-wise K folds on the operand
    (q * s_g, then add q . z_g, for the tokens of group g).  PV contracts over
    tokens: token-wise V folds on the operand P (p_l * s_l, plus sum_l p_l z_l,
    for the channels of each group); channel-wise V folds on the accumulator,
    one token group at a time (s_g * (p_g @ code_g) + z_g * sum(p_g)) because
    partial products across group boundaries cannot be accumulated unscaled
    ([SUM] 限界と未検証の範囲: accumulator folds are applied per quantization
    group).  [ABS] states the result equals the dequantized attention in
    exact arithmetic.

    kc, vc: logical codes [B, Hkv, Lcap, D]; ks/kz/vs/vz: [B, Hkv, nblk,
    128 * D / G] as stored (see quantize_sequence); G follows from their size.
    """
    q = np.asarray(q, np.float64)
    B, Hq, D = q.shape
    Hkv = kc.shape[1]
    G = Hq // Hkv
    gk = BLOCK_TOKENS * D // ks.shape[3]   # group size of K
    gv = BLOCK_TOKENS * D // vs.shape[3]   # group size of V
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.full((B, Hq), -np.inf, np.float64)
    for b in range(B):
        n = int(seq_lens[b])
        if n == 0:
            continue
        nblk = num_blocks(n)
        for h in range(Hq):
            kv = h // G
            qh = q[b, h]
            S = np.zeros(n, np.float64)
            for j in range(nblk):
                l0, l1 = j * BLOCK_TOKENS, min(n, (j + 1) * BLOCK_TOKENS)
                codes = kc[b, kv, l0:l1].astype(np.float64)          # [nv, D]
                sb = ks[b, kv, j].astype(np.float64)
                zb = kz[b, kv, j].astype(np.float64)
                if k_scheme == TOKENWISE:   # channel groups: [token][group]
                    s_tg = sb.reshape(BLOCK_TOKENS, D // gk)[:l1 - l0]
                    z_tg = zb.reshape(BLOCK_TOKENS, D // gk)[:l1 - l0]
                    for g in range(D // gk):
                        ch = slice(g * gk, (g + 1) * gk)
                        acc = codes[:, ch] @ qh[ch]                   # partial q . code of group g
                        S[l0:l1] += s_tg[:, g] * acc + z_tg[:, g] * qh[ch].sum()  # accumulator fold
                else:                       # token groups: [group][channel]
                    s_gc = sb.reshape(BLOCK_TOKENS // gk, D)
                    z_gc = zb.reshape(BLOCK_TOKENS // gk, D)
                    for g in range(BLOCK_TOKENS // gk):
                        t0, t1 = g * gk, min(l1 - l0, (g + 1) * gk)
                        if t0 >= t1:
                            continue
                        q_fold = qh * s_gc[g]                          # operand fold
                        S[l0 + t0:l0 + t1] = codes[t0:t1] @ q_fold + qh @ z_gc[g]
            S *= sm_scale
            m = S.max()
            p = np.exp(S - m)
            den = p.sum()
            acc_o = np.zeros(D, np.float64)
            for j in range(nblk):
                l0, l1 = j * BLOCK_TOKENS, min(n, (j + 1) * BLOCK_TOKENS)
                codes = vc[b, kv, l0:l1].astype(np.float64)
                pg = p[l0:l1]
                sb = vs[b, kv, j].astype(np.float64)
                zb = vz[b, kv, j].astype(np.float64)
                if v_scheme == TOKENWISE:   # channel groups: [token][group]
                    s_tg = sb.reshape(BLOCK_TOKENS, D // gv)[:l1 - l0]
                    z_tg = zb.reshape(BLOCK_TOKENS, D // gv)[:l1 - l0]
                    for g in range(D // gv):
                        ch = slice(g * gv, (g + 1) * gv)
                        acc_o[ch] += (pg * s_tg[:, g]) @ codes[:, ch] + pg @ z_tg[:, g]  # operand fold on P
                else:                       # token groups: [group][channel]
                    s_gc = sb.reshape(BLOCK_TOKENS // gv, D)
                    z_gc = zb.reshape(BLOCK_TOKENS // gv, D)
                    for g in range(BLOCK_TOKENS // gv):
                        t0, t1 = g * gv, min(l1 - l0, (g + 1) * gv)
                        if t0 >= t1:
                            continue
                        pk = pg[t0:t1]
                        acc_o += s_gc[g] * (pk @ codes[t0:t1]) + z_gc[g] * pk.sum()  # per-group accumulator fold
            out[b, h] = acc_o / den
            lse[b, h] = m + math.log(den)
    return out, lse


# ---------------------------------------------------------------------------
# Split-KV log-sum-exp merge
# ---------------------------------------------------------------------------

def merge(o_parts, lse_parts):
    """Combine partial results over disjoint token ranges.

    o_parts fp64 [R, S, D] (each normalised over its own range), lse_parts
    [R, S] (natural log; -inf marks an empty part).
    lse = log sum_s exp(lse_s); out = sum_s exp(lse_s - lse) * o_s.
    """
    o_parts = np.asarray(o_parts, np.float64)
    lse_parts = np.asarray(lse_parts, np.float64)
    R, S, D = o_parts.shape
    out = np.zeros((R, D), np.float64)
    lse = np.full(R, -np.inf, np.float64)
    for r in range(R):
        m = lse_parts[r].max()
        if m == -np.inf:
            continue
        w = np.exp(lse_parts[r] - m)
        tot = w.sum()
        out[r] = (w[:, None] * o_parts[r]).sum(axis=0) / tot
        lse[r] = m + math.log(tot)
    return out, lse


# ---------------------------------------------------------------------------
# Convenience: quantize + pack + reference outputs for a whole problem
# ---------------------------------------------------------------------------

def reference_decode(q_bits, k, v, seq_lens, bits, k_scheme, v_scheme,
                     page_table=None, num_pages=None, sm_scale=None, group=GROUP):
    """End to end on the CPU: pack K and V (groups of G elements), read the
    packed cache back, and attend over the dequantized cache.  Returns a dict
    with the packed arrays and out/lse."""
    B, Hkv, Lcap, D = k.shape
    kcodes, ks, kz = pack_cache(k, seq_lens, bits, k_scheme, K_CACHE, page_table, num_pages, group)
    vcodes, vs, vz = pack_cache(v, seq_lens, bits, v_scheme, V_CACHE, page_table, num_pages, group)
    kc, kss, kzz = unpack_cache(kcodes, ks, kz, seq_lens, bits, K_CACHE, Lcap, page_table)
    vc, vss, vzz = unpack_cache(vcodes, vs, vz, seq_lens, bits, V_CACHE, Lcap, page_table)
    khat = dequantize(kc, kss, kzz, seq_lens, k_scheme)
    vhat = dequantize(vc, vss, vzz, seq_lens, v_scheme)
    q = bf16_bits_to_f64(q_bits)
    out, lse = attend(q, khat, vhat, seq_lens, sm_scale)
    return dict(k_codes=kcodes, k_scale=ks, k_zero=kz, v_codes=vcodes, v_scale=vs,
                v_zero=vz, out=out, lse=lse, khat=khat, vhat=vhat, q=q)
