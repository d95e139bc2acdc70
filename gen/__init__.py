"""Seeded synthetic inputs for tree verification (Medusa/EAGLE-style speculative decoding).

This package is shared by the CPU oracle's tests, the GPU parity tests and the benchmark.
It only *creates* inputs: query/key/value tensors, hidden states, the LM-head weight, draft
trees (parent arrays), drafted tokens and draft distributions.  It contains none of the
verification arithmetic (tree attention, the LM-head statistics, acceptance, path selection or
KV compaction); those live in ``oracle/`` (CPU, fp64) and in the CUDA library.

The drafter itself (the Medusa heads / EAGLE draft head of "multi-token prediction
(Medusa/EAGLE)", section on Medusa, and of the jisaku glossary "Medusa", architecture table) is
outside the verified path.  Here it is simulated: a draft proposal is a noisy copy of the
target's logits, so that the synthetic trees have a realistic mix of accepted and rejected
candidates.
"""

from .bf16 import f32_to_bf16_bits, bf16_bits_to_f32, bf16_bits_to_f64  # noqa: F401
from .configs import CONFIGS, config_by_id  # noqa: F401
from .inputs import Case, compact_draft, make_config_case, make_case  # noqa: F401
from . import trees  # noqa: F401
