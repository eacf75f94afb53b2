"""fp64 CPU oracle for document-masked (varlen) attention, LSE merge and the
seq->head permutation.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
this package.  The CUDA library never calls it and shares no code with it:
no kernels, headers, helpers, tables or pre/post-processing.  Inputs reach it
as numpy arrays from the seeded generator module.

Each function restates the plain definition it computes (no tiling, no
online softmax, no fusion), citing the page passage it follows:

* ``attention.attn_fwd`` / ``attn_fwd_rows`` -- scaled dot-product attention
  (BASP, Sec. II-A "Scaled Dot-Product Attention"; HSAP, Sec. 2.2.1) inside
  each packed document only (HSAP, Sec. 2.1 "Sequence Packing": attention is
  computed only within each segment given cumulative lengths; NSP, Sec. 2.2:
  tokens of different sequences do not attend to one another), optionally
  restricted to a query range and a key range (the per-block partial of
  ring-style InterSP, HSAP Sec. 2.2.1 and Sec. 3.2 "Partition attention
  computation blocks").
* ``attention.attn_bwd`` and the sampled variants -- the analytic gradients of
  that definition (the backward pass that recomputation re-runs, NSP Sec. 2.3).
* ``attention.attn_bwd_block`` -- one ring block's share of those gradients
  (queries of one range against keys of another, probabilities normalised
  over the full row; HSAP Sec. 2.2.1 ring InterSP).
* ``merge.lse_merge`` -- combining partial results over key chunks, the
  "rescale" of ring attention's online accumulation (HSAP Sec. 2.2.1 and
  Limitations).
* ``permute.seq2head`` / ``head2seq`` -- the IntraSP all-to-all layout move
  from R^{n x H x d} per rank to R^{N x h x d}, h = H/P (HSAP Sec. 2.2.2;
  BASP Sec. II-C "DeepSpeed Ulysses").

Parity pins: every function here is checked by ``tests/test_oracle_*.py``
against closed forms, invariants, library special cases and finite
differences; none is "parity unpinned".
"""
from .attention import (allowed_interval, attn_fwd, attn_fwd_rows, attn_probs,
                        attn_bwd, attn_bwd_block, attn_bwd_dq_rows, attn_bwd_dkv_rows)
from .merge import lse_merge
from .permute import seq2head, head2seq, seq2head_groups, head2seq_groups

__all__ = [
    "allowed_interval", "attn_fwd", "attn_fwd_rows", "attn_probs", "attn_bwd", "attn_bwd_block",
    "attn_bwd_dq_rows", "attn_bwd_dkv_rows", "lse_merge", "seq2head", "head2seq",
    "seq2head_groups", "head2seq_groups",
]
