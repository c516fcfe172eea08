"""Parity at the full workload sizes, in the launch configuration bench.py
times (default grid, one call over the whole batch), on sampled outputs.

The whole cache is packed on the GPU from the seeded generators (as bench.py
does); for a sample of (sequence, kv head) units the same pre-quantization
values are drawn again, handed to the oracle, which packs, dequantizes and
attends in fp64, and the unit's query heads (4, or 8 per KV head) are
compared with the decode output.  Tolerances as in the other parity tests.
"""
import numpy as np
import pytest
import torch

import bench
import kvq_synth as synth
from oracle import kvq_oracle as orc
from tests.kvq_testlib import LSE_TOL, TOL

pytestmark = pytest.mark.gpu

SEED = 1
N_SAMPLES = 32  # seeded (sequence, kv head) units per configuration


def _sample_units(w, lens, seed):
    """First and last unit, the longest and shortest sequence, and random others."""
    g = np.random.default_rng(seed)
    units = {(0, 0), (w.batch - 1, w.num_kv_heads - 1)}
    ln = lens.tolist()
    units.add((int(np.argmax(ln)), int(g.integers(w.num_kv_heads))))
    units.add((int(np.argmin(ln)), int(g.integers(w.num_kv_heads))))
    while len(units) < N_SAMPLES:
        units.add((int(g.integers(w.batch)), int(g.integers(w.num_kv_heads))))
    return sorted(units)


def _oracle_unit(w, c, b, h, ks, vs, dev):
    n = int(c["lens_cpu"][b])
    cs = synth.outlier_channels(w, SEED, dev)
    k = synth.kv_unit(w, SEED, 0, b, h, n, dev, cs[h]).cpu().numpy()[None, None]
    v = synth.kv_unit(w, SEED, 1, b, h, n, dev).cpu().numpy()[None, None]
    g = w.num_q_heads // w.num_kv_heads
    qb = c["q"][b:b + 1, g * h:g * h + g].cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    ref = orc.reference_decode(qb, k, v, np.array([n], dtype=np.int32), w.bits, ks, vs, None, (n + 127) // 128,
                               group=w.group)
    return ref["out"][0], ref["lse"][0]


@pytest.mark.parametrize("wl,ks,vs", [
    ("b128_l32k_int4", 1, 0),
    ("b128_l32k_int4", 0, 1),
    ("b128_l32k_int4_q8", 1, 0),
    ("b128_l32k_int2_q8", 0, 0),
    ("b128_l32k_int2", 0, 0),
    ("b128_l32k_int2", 0, 1),
    ("b128_l32k_int2", 1, 0),
    ("b128_l32k_int2", 1, 1),
    ("paged_ragged_int2", 1, 0),
    ("paged_ragged_int2", 0, 0),
    ("b32_l32k_d256_g64_int4", 1, 0),
    ("b32_l32k_d128_g32_int2", 1, 0),
    ("b32_l32k_d64_g32_int2", 1, 0),
    ("b32_l32k_d64_g32_int2", 0, 1),
])
def test_full_size_sampled_units(wl, ks, vs):
    import bit_quantized_kv_decode_gb300 as kvq
    dev = torch.device("cuda")
    if wl.endswith("_q8"):  # 8 query heads per KV head
        w = synth.WORKLOADS[wl[:-3]]
        w = synth.shrink(w, num_q_heads=8 * w.num_kv_heads, name=wl)
    else:
        w = synth.WORKLOADS[wl]
    g = w.num_q_heads // w.num_kv_heads
    c = bench.build_cache(w, SEED, dev, ks, vs)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = kvq.decode_attn(c["desc"], c["q"], c["k"], c["v"], c["lens"], c["pt"], c["max_blocks"],
                               dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for b, h in _sample_units(w, c["lens_cpu"], SEED + 17):
        ro, rl = _oracle_unit(w, c, b, h, ks, vs, dev)
        ref_o.append(ro)
        ref_l.append(rl)
        got_o.append(out[b, g * h:g * h + g].double().cpu().numpy())
        got_l.append(lse[b, g * h:g * h + g].double().cpu().numpy())
    ref_o, ref_l, got_o, got_l = map(np.stack, (ref_o, ref_l, got_o, got_l))
    rms = float(np.sqrt((ref_o ** 2).mean()))
    err = float(np.abs(got_o - ref_o).max()) / rms
    lerr = float(np.abs(got_l - ref_l).max())
    print(f"[parity] {wl} k={ks} v={vs} full size, {len(ref_o)} sampled units: "
          f"max|out-oracle|/rms={err:.3e} max|lse-oracle|={lerr:.3e}")
    assert err <= TOL[0], err
    assert lerr <= LSE_TOL[0], lerr
    del c
    torch.cuda.empty_cache()
