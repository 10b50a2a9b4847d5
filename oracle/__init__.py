"""CPU oracle for the latent-MoE layer: plain, slow, fp64 — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import or run anything in this package.  The product path
(the CUDA library and its Python binding) never imports it, and this package
imports nothing from the product: the two share no code, only the seeded
input generator in ``synth``.

Modules
  nvfp4   E2M1 / E4M3 decoding tables from the format definitions, exact
          dequantisation, and the NVFP4 quantiser by definition.
  moe     the layer step by step (D, router, top-k + softmax, permutation,
          SwiGLU experts, shared expert, combine, U) and the post-norm stack.
  record  a reader of the packed expert record, written from the layout the
          library's header documents (pins the packer byte for byte).
  compare tolerances and routing-flip rule of the parity checks, the per-layer
          teacher-forced comparison and the teacher-forced stack chain (used by
          the tests and by the bench's parity report).

Parity status: the decoders, top-k, weights, permutation, SwiGLU, RMSNorm and
the record reader are pinned by tests against definitions, brute force and
library routines (tests/test_oracle_*.py).  The end-to-end layer has no
published worked example: it is pinned only through invariants (shared-expert
path with zeroed routed experts, token permutation invariance, reduction of
each step to a library routine).
"""
