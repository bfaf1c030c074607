"""Seeded synthetic workload generators (inputs only; no method arithmetic)."""
from .synth import (FULL, SMALL, SENTINEL_BYTE, Step, Workload, describe, elem_bytes,  # noqa: F401
                    chunked_prefill_spec, long_context, mixed_step, page_scales, pure_decode,
                    shared_prefix, storage_np_dtype, toy_r1r2)
