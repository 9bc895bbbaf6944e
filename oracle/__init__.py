"""fp64 CPU oracle for verify attention — test infrastructure only.

Importable by ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py``; never by the library itself.
"""
from .verify_oracle import *  # noqa: F401,F403
from .verify_oracle import (ancestors, attend, decode_bf16, decode_fp16, dequant_q8_0,
                            gather_index, merge, partial, row_map, row_masks,
                            split_ranges, verify_attention, verify_case,
                            visible_positions)
