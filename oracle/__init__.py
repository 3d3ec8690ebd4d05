"""CPU oracle for one selectively batched Transformer iteration (Orca).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference arm may import this package.  The
CUDA path never calls it, and it shares no code with the CUDA path: the only
module both sides use is ``synth`` (seeded inputs, no arithmetic of the
method).

What it computes, and from which passage:

* ``model``     - a GPT decoder that generates each request alone, one token
                  at a time, with a per-request K/V cache.  Selective batching
                  must reproduce exactly this ("continuous-batched output
                  equals per-request generation": CS349D Lecture 2, sections
                  4.1 and 4.2; the batched-vs-individual check in section 4.2).
* ``scheduler`` - Algorithm 1 (ORCA scheduling algorithm) with
                  n_workers = 1: FCFS ``Select`` with max_bs and max_tokens
                  reservation, plus a contiguous first-fit K/V slot pool
                  (Orca walk-through, "两个约束：max batch size 与 GPU 显存").
* ``ragged``    - the flattened [sum L_i, H] row layout of Figure 5 and the
                  useful/padded row and (query, key) pair counts of
                  CS349D Lecture 2, Exercise 4.
* ``numerics``  - bf16 round-to-nearest-even, LayerNorm, tanh-GeLU, softmax.

Floating point runs in numpy float64.  In bf16 mode the oracle rounds to
bf16 exactly where the CUDA path stores bf16 (LayerNorm outputs, Q/K/V,
attention output, GeLU output); the residual stream stays wide.

Parity status: the integer parts are pinned by the pages' worked examples
(Figure 5, the demo-4 timeline, Exercise 4, the break rule).  The forward
math is pinned by an independent full-sequence forward built from torch
library routines (layer_norm, linear, scaled_dot_product_attention, gelu)
and by closed-form special cases; the logits of the random-init models have
no printed values on the pages.
"""
