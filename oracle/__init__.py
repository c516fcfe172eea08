"""CPU oracle for quantized-KV decode attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU baseline / reference
arm of ``bench.py`` may import this package.
"""
from . import kvq_oracle  # noqa: F401
