"""C-ABI checks that need no GPU: the library builds, loads and exports every
symbol include/kvq.h declares, and host-side validation rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest
import torch

import __graft_entry__ as entry
from bit_quantized_kv_decode_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    entry.build()
    return _lib.load()


def _header_symbols():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    return sorted(set(re.findall(r"KVQ_API\s+[\w\s\*]+?\b(kvq_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    declared = _header_symbols()
    assert len(declared) >= 8
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(_lib.EXPORTS) == declared


def test_only_declared_symbols_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.lib_path()], capture_output=True, text=True).stdout
    exported = sorted(l.split()[-1] for l in out.splitlines() if " T " in l)
    assert exported == _header_symbols()


def test_status_strings_and_version(lib):
    assert lib.kvq_status_string(0) == b"ok"
    assert lib.kvq_status_string(3) == b"workspace too small"
    assert lib.kvq_status_string(99) == b"unknown status"
    assert lib.kvq_version() >= 100


def _cache(bits=4, k=0, v=1, heads=8, pages=1024, hd=128, group=0):
    return _lib.CacheDesc(bits, k, v, hd, heads, pages, group)


def test_cache_bytes(lib):
    cb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.kvq_cache_bytes(ctypes.byref(_cache(4)), ctypes.byref(cb), ctypes.byref(sb)) == 0
    assert cb.value == 1024 * 8 * 8192 and sb.value == 1024 * 8 * 128 * 2
    assert lib.kvq_cache_bytes(ctypes.byref(_cache(2)), ctypes.byref(cb), ctypes.byref(sb)) == 0
    assert cb.value == 1024 * 8 * 4096
    assert lib.kvq_cache_bytes(ctypes.byref(_cache(3)), ctypes.byref(cb), ctypes.byref(sb)) == 2
    # head dims 64 / 256 and groups of 32 / 64: codes 128 * D * b / 8, s / z 128 * D / G per page and head
    assert lib.kvq_cache_bytes(ctypes.byref(_cache(4, hd=256, group=64)), ctypes.byref(cb), ctypes.byref(sb)) == 0
    assert cb.value == 1024 * 8 * 128 * 256 * 4 // 8 and sb.value == 1024 * 8 * (128 * 256 // 64) * 2
    assert lib.kvq_cache_bytes(ctypes.byref(_cache(2, hd=64, group=32)), ctypes.byref(cb), ctypes.byref(sb)) == 0
    assert cb.value == 1024 * 8 * 128 * 64 * 2 // 8 and sb.value == 1024 * 8 * (128 * 64 // 32) * 2
    for hd, group in ((64, 0), (64, 128), (96, 32), (128, 16), (128, 96), (512, 128)):
        assert lib.kvq_cache_bytes(ctypes.byref(_cache(4, hd=hd, group=group)), ctypes.byref(cb),
                                   ctypes.byref(sb)) == 2, (hd, group)
    assert lib.kvq_cache_bytes(None, ctypes.byref(cb), ctypes.byref(sb)) == 1


def test_workspace_size_host_only(lib):
    # a small call (8 x 8 x 32 triples of (sequence, kv head, block)): the specialised kernel
    d = _lib.AttnDesc(_cache(4, 1, 0, pages=8 * 32), 8, 32, 32, 0, 0.0, 304, 0)
    n = ctypes.c_size_t()
    assert lib.kvq_decode_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 0
    # counters (one per sequence x kv head) + part lse + part out, each 256-byte aligned
    assert n.value == 8 * 8 * 4 + 304 * 2 * 4 * 4 + 304 * 2 * 4 * 128 * 4
    bad = _lib.AttnDesc(_cache(4), 128, 24, 256, 0, 0.0, 304, 0)  # 3 query heads per KV head: not built
    assert lib.kvq_decode_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == 2
    bad = _lib.AttnDesc(_cache(4), 128, 20, 256, 0, 0.0, 304, 0)  # not a multiple of the KV heads
    assert lib.kvq_decode_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == 2
    for hq in (8, 16):  # 1 and 2 query heads per KV head: one unit per KV head
        d = _lib.AttnDesc(_cache(4, pages=8 * 32), 8, hq, 32, 0, 0.0, 304, 0)
        assert lib.kvq_decode_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 0
        assert n.value == 8 * 8 * 4 + 304 * 2 * 4 * 4 + 304 * 2 * 4 * 128 * 4
    d = _lib.AttnDesc(_cache(4, pages=8 * 32), 8, 64, 32, 0, 0.0, 304, 0)  # 8, small call: two units per KV head
    assert lib.kvq_decode_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 0
    assert n.value == 8 * 16 * 4 + 304 * 2 * 4 * 4 + 304 * 2 * 4 * 128 * 4
    bad = _lib.AttnDesc(_cache(4), 0, 32, 256, 0, 0.0, 304, 0)
    assert lib.kvq_decode_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == 1
    bad = _lib.AttnDesc(_cache(4), 2048, 32, 256, 0, 0.0, 304, 0)
    assert lib.kvq_decode_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == 2
    bad = _lib.AttnDesc(_cache(4), 8, 32, 256, 7, 0.0, 304, 0)
    assert lib.kvq_decode_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == 1


def test_e2m1_flag_validation(lib):
    """The E2M1 V placement is built for 2-bit caches, FP8 operands and 4
    query heads per KV head; other combinations and unknown flag bits are
    rejected on the host."""
    n = ctypes.c_size_t()
    ok = _lib.AttnDesc(_cache(2, 1, 0), 8, 32, 32, 0, 0.0, 304, _lib.FLAG_E2M1_V)
    assert lib.kvq_decode_workspace_size(ctypes.byref(ok), ctypes.byref(n)) == 0
    for d in (_lib.AttnDesc(_cache(4, 1, 0), 8, 32, 32, 0, 0.0, 304, _lib.FLAG_E2M1_V),   # 4-bit codes
              _lib.AttnDesc(_cache(2, 1, 0), 8, 32, 32, 1, 0.0, 304, _lib.FLAG_E2M1_V),   # BF16 operands
              _lib.AttnDesc(_cache(2, 1, 0), 8, 64, 32, 0, 0.0, 304, _lib.FLAG_E2M1_V),   # 8 query heads per KV head
              _lib.AttnDesc(_cache(2, 1, 0), 8, 16, 32, 0, 0.0, 304, _lib.FLAG_E2M1_V)):  # 2 query heads per KV head
        assert lib.kvq_decode_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 2
    bad = _lib.AttnDesc(_cache(2, 1, 0), 8, 32, 32, 0, 0.0, 304, 0x8)  # unknown flag bit
    assert lib.kvq_decode_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == 1
    hook = _lib.AttnDesc(_cache(2, 1, 0), 8, 32, 32, 0, 0.0, 304, _lib.FLAG_TEST_STALL_MMA)  # the MMA stall test hook
    assert lib.kvq_decode_workspace_size(ctypes.byref(hook), ctypes.byref(n)) == 0


def _general_ws(batch, units, splits, gq, head_dim):
    """Workspace of the general kernel, each part 256-byte aligned: the plan's
    prefix (batch + 1 ints), one 16-byte assignment per CTA, and one part slot
    per CTA holding gq heads' lse and outputs; CTAs = the plan's target
    (units x ranges) plus one per unit."""
    r256 = lambda x: (x + 255) // 256 * 256
    slots = units * splits + units
    return r256((batch + 1) * 4) + r256(slots * 16) + r256(slots * gq * 4) + r256(slots * gq * head_dim * 4)


def test_general_geometry_workspace_host_only(lib):
    """Head dims 64 / 256 and groups of 32 / 64 take the block-range kernel;
    its target is ranges = ceil(num_ctas / units) per unit, capped at
    max_blocks; both operand modes; not the E2M1 V placement."""
    n = ctypes.c_size_t()
    d = _lib.AttnDesc(_cache(4, 1, 0, hd=256, group=64, pages=16 * 64), 16, 32, 64, 0, 0.0, 304, 0)
    assert lib.kvq_decode_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 0
    assert n.value == _general_ws(16, 16 * 8, 3, 4, 256)  # 128 units, 304 CTAs wanted -> 3 ranges
    d = _lib.AttnDesc(_cache(2, 0, 1, hd=64, group=32, pages=16 * 64), 2, 16, 2, 0, 0.0, 100000, 0)
    assert lib.kvq_decode_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 0
    assert n.value == _general_ws(2, 2 * 8, 2, 2, 64)  # two ranges at most (max_blocks = 2); 2 heads per unit
    bf16 = _lib.AttnDesc(_cache(2, 1, 0, hd=128, group=32), 8, 32, 32, 1, 0.0, 304, 0)
    assert lib.kvq_decode_workspace_size(ctypes.byref(bf16), ctypes.byref(n)) == 0
    # the BF16-operand mode takes the block-range kernel on every geometry
    bf16 = _lib.AttnDesc(_cache(4, 1, 0, pages=16 * 64), 16, 32, 64, 1, 0.0, 304, 0)
    assert lib.kvq_decode_workspace_size(ctypes.byref(bf16), ctypes.byref(n)) == 0
    assert n.value == _general_ws(16, 16 * 8, 3, 4, 128)
    # 8 query heads per KV head: one 8-head unit per KV head
    h8 = _lib.AttnDesc(_cache(4, 1, 0, hd=64, group=64, pages=16 * 64), 16, 64, 64, 0, 0.0, 304, 0)
    assert lib.kvq_decode_workspace_size(ctypes.byref(h8), ctypes.byref(n)) == 0
    assert n.value == _general_ws(16, 16 * 8, 3, 8, 64)
    bad = _lib.AttnDesc(_cache(2, 1, 0, hd=128, group=32), 8, 32, 32, 0, 0.0, 304, _lib.FLAG_E2M1_V)
    assert lib.kvq_decode_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == 2


def _spec_ws(batch, units, ctas):
    """Workspace of the specialised kernel, each part 256-byte aligned:
    arrival counters (one int per unit), part lse and part outputs (two parts
    of 4 heads per CTA)."""
    r256 = lambda x: (x + 255) // 256 * 256
    return r256(batch * units * 4) + r256(ctas * 2 * 4 * 4) + r256(ctas * 2 * 4 * 128 * 4)


def test_default_geometry_routing_host_only(lib):
    """E4M3 operands at head dim 128, groups of 128: every call holding at
    least 8,192 (sequence, unit, block) triples of max_blocks per unit takes
    the general kernel, whatever its scheme pair and query heads per KV head;
    smaller calls and the E2M1 V placement take the specialised kernel.  Read
    from kvq_decode_path and from the workspace each layout needs."""
    n = ctypes.c_size_t()
    path = ctypes.c_int32()
    for bits in (2, 4):
        for k in (0, 1):
            for v in (0, 1):
                for hq in (8, 16, 32, 64):
                    g = hq // 8
                    d = _lib.AttnDesc(_cache(bits, k, v, pages=128 * 256), 128, hq, 256, 0, 0.0, 304, 0)
                    assert lib.kvq_decode_path(ctypes.byref(d), ctypes.byref(path)) == 0
                    assert path.value == _lib.PATH_GENERAL, (bits, k, v, hq)
                    assert lib.kvq_decode_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 0
                    units = 8 * 128  # one unit per KV head (8 heads: one 8-head unit)
                    assert n.value == _general_ws(128, units, 1, 8 if g == 8 else min(g, 4), 128), (bits, k, v, hq)
    # the threshold: 32 x 16 units x 16 blocks = 8,192 triples (8 heads) -> general, one block less -> specialised
    for mb, want in ((16, _lib.PATH_GENERAL), (15, _lib.PATH_SPECIALISED)):
        d = _lib.AttnDesc(_cache(2, 1, 0, pages=32 * 16), 32, 64, mb, 0, 0.0, 304, 0)
        assert lib.kvq_decode_path(ctypes.byref(d), ctypes.byref(path)) == 0 and path.value == want, mb
    # a small call (8 x 8 x 32 = 2,048 triples) stays specialised
    for bits, k, v in ((2, 0, 0), (4, 1, 0)):
        d = _lib.AttnDesc(_cache(bits, k, v, pages=8 * 32), 8, 32, 32, 0, 0.0, 304, 0)
        assert lib.kvq_decode_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 0
        assert n.value == _spec_ws(8, 8, 304)
        assert lib.kvq_decode_path(ctypes.byref(d), ctypes.byref(path)) == 0
        assert path.value == _lib.PATH_SPECIALISED
    # the E2M1 V placement: specialised at any size
    d = _lib.AttnDesc(_cache(2, 0, 0, pages=128 * 256), 128, 32, 256, 0, 0.0, 304, _lib.FLAG_E2M1_V)
    assert lib.kvq_decode_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 0
    assert n.value == _spec_ws(128, 8, 304)
    assert lib.kvq_decode_path(ctypes.byref(d), ctypes.byref(path)) == 0 and path.value == _lib.PATH_SPECIALISED
    # other geometries and the BF16 mode: general at any size; bad descriptors are refused
    for d in (_lib.AttnDesc(_cache(4, 1, 0, hd=256, group=64, pages=64), 2, 32, 4, 0, 0.0, 304, 0),
              _lib.AttnDesc(_cache(2, 1, 0, pages=64), 2, 32, 4, 1, 0.0, 304, 0)):
        assert lib.kvq_decode_path(ctypes.byref(d), ctypes.byref(path)) == 0 and path.value == _lib.PATH_GENERAL
    bad = _lib.AttnDesc(_cache(4), 128, 24, 256, 0, 0.0, 304, 0)  # 3 query heads per KV head
    assert lib.kvq_decode_path(ctypes.byref(bad), ctypes.byref(path)) == 2
    assert lib.kvq_decode_path(ctypes.byref(d), None) == 1


def test_validation_precedes_device(lib):
    """Bad arguments are rejected on the host (no device needed)."""
    c = _cache(4)
    P = ctypes.c_void_p
    fake = P(0x10000)  # never dereferenced: validation fails first
    # which out of range
    assert lib.kvq_pack(ctypes.byref(c), 2, fake, 1, 128, None, None, 1, fake, fake, fake, None, None) == 1
    # misaligned x
    assert lib.kvq_pack(ctypes.byref(c), 0, P(0x10004), 1, 128, None, None, 1, fake, fake, fake, None, None) == 1
    # max_blocks too small for max_seq_len
    assert lib.kvq_pack(ctypes.byref(c), 0, fake, 1, 300, None, None, 2, fake, fake, fake, None, None) == 1
    # contiguous cache larger than num_pages
    small = _cache(4, pages=3)
    assert lib.kvq_pack(ctypes.byref(small), 0, fake, 2, 256, None, None, 2, fake, fake, fake, None, None) == 1
    # decode: null output
    d = _lib.AttnDesc(c, 1, 32, 2, 0, 0.0, 1, 0)
    args = [fake] * 7 + [fake, None, None, fake, fake, 1 << 20, None, None]
    assert lib.kvq_decode_attn(ctypes.byref(d), *args) == 1
    # merge: bad head_dim
    assert lib.kvq_merge(fake, fake, 4, 2, 130, fake, fake, None) == 1
    # append: which out of range, missing window, misaligned x_new, contiguous cache too small
    app = [fake, 1, fake, fake, 2, fake, fake, fake, fake, None, None]
    assert lib.kvq_append(ctypes.byref(c), 2, *app) == 1
    assert lib.kvq_append(ctypes.byref(c), 0, fake, 1, fake, fake, 2, None, fake, fake, fake, None, None) == 1
    assert lib.kvq_append(ctypes.byref(c), 0, P(0x10004), 1, fake, fake, 2, fake, fake, fake, fake, None, None) == 1
    assert lib.kvq_append(ctypes.byref(small), 0, fake, 2, fake, None, 2, fake, fake, fake, fake, None, None) == 1


def test_no_device_reports_device_error(lib):
    """On a machine without a GPU a well-formed call fails loudly (no fallback)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    c = _cache(4)
    fake = ctypes.c_void_p(0x10000)
    assert lib.kvq_pack(ctypes.byref(c), 0, fake, 1, 128, None, None, 1, fake, fake, fake, None, None) == 5


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-only: on a GPU machine the call would launch")
def test_static_entry_routes_within_its_scratch_host_only(lib):
    """The static entry's 4 MiB scratch: a call the general kernel would take
    with a larger workspace goes to the specialised kernel when that one takes
    it (E4M3, head dim 128, groups of 128) -- the call then passes the scratch
    check and stops at the device check (no GPU here) -- and is refused with
    KVQ_ERR_WORKSPACE when it does not (BF16 operands)."""
    fake = ctypes.c_void_p(0x10000)
    n = ctypes.c_size_t()
    d = _lib.AttnDesc(_cache(2, 0, 0, pages=128 * 256), 128, 32, 256, 0, 0.0, 304, 0)
    assert lib.kvq_decode_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 0 and n.value > 4 << 20
    assert lib.kvq_decode_attn_static(ctypes.byref(d), *([fake] * 7), fake, None, fake, fake, None, None) == 5
    bf16 = _lib.AttnDesc(_cache(2, 0, 0, pages=128 * 256), 128, 32, 256, 1, 0.0, 304, 0)
    assert lib.kvq_decode_attn_static(ctypes.byref(bf16), *([fake] * 7), fake, None, fake, fake, None, None) == 3
