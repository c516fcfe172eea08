"""Host-side checks of the general kernel's launch-shape rules
(`csrc/decode_general.h`): for every instance the library builds (head dim,
group size, bit width, scheme pair, operand mode, query heads per unit), the
resident-CTA count it plans must fit the SM -- tensor-memory columns and
shared memory (the copy ring, Q', P' and scratch, plus the per-CTA
reservation) -- the channel-halves-in-turn layout must be taken exactly where
it raises residency, and the layout must keep its regions in order.  The
rules are compiled as host code from the header itself (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "bit_quantized_kv_decode_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "decode_general.h"
using namespace kvq;
int main() {
  for (int bf = 0; bf < 2; ++bf)
    for (int nh = 4; nh <= 8; nh += 4)
      for (int D : {64, 128, 256})
        for (int G : {32, 64, 128})
          for (int bits : {2, 4})
            for (int kc = 0; kc < 2; ++kc)
              for (int vc = 0; vc < 2; ++vc) {
                if (G > D) continue;
                const bool turn = gen_turn(bits, D, G, kc, vc, bf, nh);
                const int st = gen_single_stage(bits, D, G, kc, vc, bf, nh) ? 1 : 2;
                const GenLayout l = gen_layout(bits, D, G, kc, vc, bf, nh, st);
                printf("%d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d\n", bf, nh, D, G, bits, kc, vc,
                       gen_ctas_per_sm(bits, D, G, kc, vc, bf, nh), gen_min_ctas(bits, D, G, kc, vc, bf, nh), st,
                       (int)turn, l.tmem_cols, l.total_bytes, l.q_off, l.p_off, l.scratch_off, l.stage_bytes,
                       (int)l.seq_halves, gen_fit(bits, D, G, kc, vc, bf, nh, 1, true),
                       gen_fit(bits, D, G, kc, vc, bf, nh, 2, false));
              }
  printf("smem %d %d scratch %d\n", kGenSmemPerSm, kGenSmemPerCta, kGenScratchBytes);
  return 0;
}
"""

FIELDS = ("bf16", "nh", "D", "G", "bits", "kcw", "vcw", "ctas", "min_ctas", "stages", "turn", "tmem_cols",
          "total_bytes", "q_off", "p_off", "scratch_off", "stage_bytes", "seq", "fit_turn1", "fit_plain2")


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else shutil.which("nvcc")


@pytest.fixture(scope="module")
def shapes(tmp_path_factory):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    d = tmp_path_factory.mktemp("shape")
    src, exe = d / "shape.cu", d / "shape"
    src.write_text(PROGRAM)
    r = subprocess.run([nvcc, "-std=c++17", "-I", CSRC, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines()
    smem = out[-1].split()
    rows = [dict(zip(FIELDS, map(int, line.split()))) for line in out[:-1]]
    return rows, int(smem[1]), int(smem[2]), int(smem[4])


def test_every_instance_fits_the_sm(shapes):
    rows, smem_per_sm, per_cta, _ = shapes
    assert len(rows) == 8 * 2 * 2 * 2 * 2 * 2  # (D, G) pairs x bits x K scheme x V scheme x operands x heads
    for r in rows:
        c = r["ctas"]
        assert 1 <= c <= (8 if r["nh"] == 4 else 6), r
        assert c * r["tmem_cols"] <= 512, r                            # tensor memory
        assert c * (r["total_bytes"] + per_cta) <= smem_per_sm, r      # shared memory at the planned ring
        assert r["total_bytes"] <= 227 * 1024, r                       # one CTA's opt-in limit
        assert r["tmem_cols"] in (32, 64, 128, 256, 512), r
        assert r["min_ctas"] == (c if r["nh"] > 4 else max(c, 4)), r  # launch bounds
        if r["nh"] > 4:
            assert c <= (6 if r["bits"] == 2 else 5), r


def test_layout_regions_in_order(shapes):
    rows, _, _, scratch = shapes
    for r in rows:
        assert r["q_off"] == r["stages"] * r["stage_bytes"], r
        assert r["q_off"] < r["p_off"] < r["scratch_off"], r
        assert r["total_bytes"] == r["scratch_off"] + scratch, r
        for off in ("q_off", "p_off", "scratch_off", "stage_bytes"):
            assert r[off] % 16 == 0, (off, r)  # 16-byte bulk-copy and vector alignment


def test_halves_in_turn_exactly_where_they_raise_residency(shapes):
    rows, _, _, _ = shapes
    for r in rows:
        if r["D"] <= 128:
            assert not r["turn"], r
            continue
        assert r["turn"] == (r["fit_turn1"] > r["fit_plain2"]), r
        if r["turn"]:
            assert r["seq"] and r["stages"] == 1 and r["ctas"] == r["fit_turn1"], r
    # the measured case: 4-bit, groups of 64, K-cw/V-tw, 4 heads, E4M3 -- 2 -> 4 CTAs per SM
    (m,) = [r for r in rows if (r["bf16"], r["nh"], r["D"], r["G"], r["bits"], r["kcw"], r["vcw"]) ==
            (0, 4, 256, 64, 4, 1, 0)]
    assert m["turn"] and m["ctas"] == 4 and m["fit_plain2"] == 2


def test_one_stage_rings_at_head_dim_128(shapes):
    rows, _, _, _ = shapes
    for r in rows:
        if r["D"] != 128:
            continue
        single = (r["bits"] == 4 and r["G"] == 128 and (r["vcw"] or not r["kcw"]) and not r["bf16"] and r["nh"] == 4)
        assert (r["stages"] == 1) == single, r
        if single:
            assert r["ctas"] == 8, r
