"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

Holds random-number generation and data placement only, none of the step's
arithmetic.
"""
from .philox import philox4x32_10, tree_uniforms, uint32_to_unit_float
from .workloads import (STATIC_SHAPE_60, WORKLOADS, Workload, attention_inputs,
                        draft_logits, draft_like_rows, kv_lengths, scaled,
                        static_template, target_logits, uniforms)
