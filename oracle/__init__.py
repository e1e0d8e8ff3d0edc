"""CPU oracle for the tensor-parallel MLP block and the vocab-parallel
cross-entropy of Megatron-LM (Shoeybi et al. 2019). TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the bench's CPU-baseline / reference
arm may import this package. The product path (the CUDA library and its Python
binding) never imports it, links it or falls back to it.

Everything here is plain float64 numpy (and scipy's ``erf``), written from the
definitions on the pages, with no blocking, fusion or reordering beyond what a
definition states. Sources, cited by page title and section:

[p1] "Megatron-LM: Training Multi-Billion Parameter Language Models Using Model
     Parallelism" (paper-graph-ui summary), §3.4 "Detailed, Sentence-Based
     Technical Breakdown": column-parallel GEMM, row-parallel GEMM, g/f
     operators, vocab-parallel input embedding, fused vocab-parallel
     cross-entropy, vocabulary padding.
[p3] "Tensor and pipeline parallelism, and choosing a layout" (ML Systems,
     lesson 9), §3 "Definitions and main results", Proposition (Megatron MLP
     split), proof steps 1-5 (forward and backward).
[p5] "Megatron-LM, annotated" (ai-primer), §2.2 (GELU, erf form), §3.1 (the
     two-token MLP example), §3.2 (attention block), §3.4 (embedding, loss,
     vocabulary padding).

The cross-entropy backward (``ce_bwd``) is not spelled out on the pages, which
train the model but describe only the forward fusion; it is the plain derivative
of the softmax cross-entropy, pinned by finite differences.

Pins (tests marked "not gpu"): GELU values printed in [p5] §2.2, the [p5] §3.1
worked example and its wrong row cut, closed forms of GELU, finite differences
of the backward, brute-force softmax cross-entropy on tiny vocabularies, the
E = 0 closed form, shift and partition invariance, and the [p5] §3.4 padding
arithmetic. Parity of the sampled-index helpers is pinned to the full oracle.
Nothing here is "parity unpinned".
"""
from .gelu import gelu, gelu_prime, std_normal_cdf, std_normal_pdf
from .mlp import (
    mlp_fwd,
    mlp_bwd,
    mlp_sharded_fwd,
    mlp_sharded_bwd,
    first_layer_row_cut,
    mlp_fwd_rows,
    mlp_bwd_sampled,
)
from .ce import (ce_loss, ce_partition_triples, ce_combine, ce_loss_partitioned, ce_bwd, ce_logsumexp,
                 ce_bwd_sampled)
from .padding import pad_vocab
from .embed import embed_sharded
from .attn import attention_heads, attn_fwd, attn_fwd_sharded, attn_fwd_rows

__all__ = [
    "gelu", "gelu_prime", "std_normal_cdf", "std_normal_pdf",
    "mlp_fwd", "mlp_bwd", "mlp_sharded_fwd", "mlp_sharded_bwd", "first_layer_row_cut",
    "mlp_fwd_rows", "mlp_bwd_sampled",
    "ce_loss", "ce_partition_triples", "ce_combine", "ce_loss_partitioned", "ce_bwd", "ce_logsumexp",
    "ce_bwd_sampled",
    "pad_vocab", "embed_sharded",
    "attention_heads", "attn_fwd", "attn_fwd_sharded", "attn_fwd_rows",
]
