"""Seeded synthetic workload generators (inputs only; no method arithmetic)."""
from .synth import (FULL, MULTI_ROW_FULL, MULTI_ROW_SMALL, SMALL, SENTINEL_BYTE,  # noqa: F401
                    Step, Workload, chunked_prefill_spec, describe, elem_bytes, long_context,
                    mixed_step, page_scales, pure_decode, shared_prefix, spec_decode,
                    storage_np_dtype, toy_r1r2)
