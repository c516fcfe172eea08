"""Diagnostic: the folded decode attention with tensor-core operand rounding.

TEST INFRASTRUCTURE (diagnostic only; never a parity target).  It predicts how
far a tensor-core implementation that feeds E4M3 or BF16 operands drifts from
the exact result, so that tolerances and operand splits can be chosen from
arithmetic rather than by trial.  It follows the folded formulation of
``kvq_oracle.attend_folded`` ([SUM] 解説: acc-fold / operand-fold) and rounds
the two non-integer operands:

  * Q' (the query, times s for channel-wise K) is scaled per head by a power
    of two so that its largest magnitude lies in [128, 256) and is then split
    into ``q_splits`` E4M3 (or BF16) parts hi + mid + lo; the sum of the parts
    is what the tensor core sees;
  * P' (the probabilities, times s for token-wise V) is scaled by a power of
    two per 128-token tile and split into ``p_splits`` parts.

The KV codes themselves are exact in E4M3 (4-bit codes as q * 2^-9) and E2M1
(2-bit codes as q / 2) ([SUM] 解説: the bit placements), so they carry no
rounding here.  Accumulation is taken as exact.
"""
from __future__ import annotations

import math

import numpy as np

from .kvq_oracle import BLOCK_TOKENS, TOKENWISE, num_blocks


def round_e4m3(x):
    """Round to the nearest E4M3 (1-4-3, bias 7, max 448) value, ties to even,
    saturating at +-448."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)                    # a = m * 2^e, m in [0.5, 1)
    E = np.maximum(e - 1, -6)             # below 2^-6 the spacing stays 2^-9
    quantum = np.ldexp(1.0, E - 3)
    r = np.minimum(np.round(a / quantum) * quantum, 448.0)
    return np.sign(x) * r


def round_bf16(x):
    """Round to the nearest bf16 value (8 significant bits), ties to even."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)
    E = np.maximum(e - 1, -126)
    quantum = np.ldexp(1.0, E - 7)
    return np.sign(x) * np.round(a / quantum) * quantum


def split(x, parts, fmt):
    """x ~= sum of ``parts`` values of format ``fmt`` (greedy residual split)."""
    rnd = round_e4m3 if fmt == "e4m3" else round_bf16
    acc = np.zeros_like(x)
    r = np.asarray(x, np.float64).copy()
    for _ in range(parts):
        p = rnd(r)
        acc += p
        r = r - p
    return acc


def pow2_scale(maxabs):
    """2^k with maxabs * 2^k in [128, 256) (1 when maxabs is 0)."""
    maxabs = np.asarray(maxabs, np.float64)
    with np.errstate(divide="ignore"):
        k = np.where(maxabs > 0, 7 - np.floor(np.log2(np.where(maxabs > 0, maxabs, 1.0))), 0.0)
    return np.ldexp(1.0, k.astype(int))


def attend_emulated(q, kc, ks, kz, vc, vs, vz, seq_lens, k_scheme, v_scheme,
                    fmt="e4m3", q_splits=3, p_splits=2, sm_scale=None):
    """Folded attention with rounded Q' and P' operands (see module doc)."""
    q = np.asarray(q, np.float64)
    B, Hq, D = q.shape
    Hkv = kc.shape[1]
    G = Hq // Hkv
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    out = np.zeros((B, Hq, D))
    lse = np.full((B, Hq), -np.inf)
    for b in range(B):
        n = int(seq_lens[b])
        if n == 0:
            continue
        nblk = num_blocks(n)
        for h in range(Hq):
            kv = h // G
            qh = q[b, h]
            m_run, l_run, o_run = -np.inf, 0.0, np.zeros(D)
            if k_scheme == TOKENWISE:
                sc = pow2_scale(np.abs(qh).max())
                q_op = split(qh * sc, q_splits, fmt) / sc
            for j in range(nblk):
                l0, l1 = j * BLOCK_TOKENS, min(n, (j + 1) * BLOCK_TOKENS)
                codes = kc[b, kv, l0:l1].astype(np.float64)
                if k_scheme == TOKENWISE:
                    s_l = ks[b, kv, j, :l1 - l0].astype(np.float64)
                    z_l = kz[b, kv, j, :l1 - l0].astype(np.float64)
                    S = s_l * (codes @ q_op) + z_l * qh.sum()
                else:
                    qf = qh * ks[b, kv, j].astype(np.float64)
                    sc = pow2_scale(np.abs(qf).max())
                    qf_op = split(qf * sc, q_splits, fmt) / sc
                    S = codes @ qf_op + qh @ kz[b, kv, j].astype(np.float64)
                S = S * sm_scale
                m_new = max(m_run, S.max())
                alpha = math.exp(m_run - m_new) if m_run > -np.inf else 0.0
                p = np.exp(S - m_new)
                vcode = vc[b, kv, l0:l1].astype(np.float64)
                if v_scheme == TOKENWISE:
                    s_l = vs[b, kv, j, :l1 - l0].astype(np.float64)
                    z_l = vz[b, kv, j, :l1 - l0].astype(np.float64)
                    sc = pow2_scale(s_l.max()) if fmt == "e4m3" else 1.0
                    p_op = split(p * s_l * sc, p_splits, fmt) / sc
                    tile_o = p_op @ vcode + p @ z_l
                else:
                    s_g = vs[b, kv, j].astype(np.float64)
                    z_g = vz[b, kv, j].astype(np.float64)
                    p_op = split(p * 256.0, p_splits, fmt) / 256.0
                    tile_o = s_g * (p_op @ vcode) + z_g * p.sum()
                o_run = o_run * alpha + tile_o
                l_run = l_run * alpha + p.sum()
                m_run = m_new
            out[b, h] = o_run / l_run
            lse[b, h] = m_run + math.log(l_run)
    return out, lse
