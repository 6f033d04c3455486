"""CPU oracle for the Oases tensor-parallel transformer block.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never calls it, and it shares no code with the CUDA library: the only thing
both sides use is the seeded input generator in ``synth/``.

Source followed throughout: the arXiv HTML of "Oases: Efficient Large-Scale
Model Training on Commodity Servers via Overlapped and Automated Tensor Model
Parallelism" (arXiv 2305.16121), cited below as "Oases" plus the section,
equation or algorithm:
  - Oases §IV-A, Fig. 4a: the operator sequence (F_i, C_i(F), F_j) of an FFN or
    attention layer under tensor model parallelism and its default recompute
    backward (R_i, C_i(R), R_j), (B_j, B_i, C_i(B)).
  - Oases §IV, Fig. 4b: two sub-batches; operators with different
    superscripts pipeline.
  - Oases §IV, Eq. (1), Fig. 4d: y = sum_i x_i over the w shards, so
    dy/dx_i = 1; fine-grained recomputation starts after communication
    operators and drops C_i(R).
  - Oases §IV, Algorithm 1: the training schedule (sub-batch split,
    Forward / StartAsync / Sync, recompute sequences without communication,
    reverse-order Recompute then Backward).
The block internals (pre-LayerNorm, erf GeLU, causal softmax attention,
residual, row-parallel bias added once after the shard sum) are not on the
pages; they follow the textbook definitions of these layers.  ``oracle.fp8``
(E4M3 rounding and MX block-scaled GEMMs, for an FP8 form of the block's
GEMMs that the pages do not describe) follows the published format
definitions cited in its header.

Everything is float64 numpy.  Parity status of each function is stated in its
docstring; every function here is pinned by a test in tests/test_oracle_*.py.
"""
from .ops import (layer_norm, layer_norm_backward, gelu, gelu_grad, attention_head,
                  attention_head_backward)
from .definition import block_forward_plain, block_loss_plain
from .schedule import run_step, build_operator_sequence, Trace

__all__ = ["layer_norm", "layer_norm_backward", "gelu", "gelu_grad", "attention_head",
           "attention_head_backward", "block_forward_plain", "block_loss_plain",
           "run_step", "build_operator_sequence", "Trace"]
