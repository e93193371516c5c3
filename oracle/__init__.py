"""CPU oracle for the packed ternary / sign-bitmap GEMMs.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the method computes, in float64 on the host.  It exists
to check the CUDA path; it is never part of it.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import it.  It shares no code with
``binary_packed_weight_gb300`` and imports nothing from it.

Modules
-------
``f16``   IEEE-754 binary16 decode written from the format definition.
``tq2``   ``BlockTQ2_0_g128`` parse / dequantize and the GEMM
          ``out[m,n] = sum_k x[m,k] * W[n,k]``.
``blr``   the binary low-rank layer ``W = diag(h) S_U diag(l) S_V^T diag(g)``:
          sign-bitmap expansion, forward and backward.

Sources (web pages, cited by title and section):

* "oxibonsai-kernels 0.2.1, src/gpu_backend/metal_graph/tests_gemm_tq2.rs"
  -- the ternary TQ2 GEMM and its block format (tests
  ``test_encode_gemm_tq2_matches_reference`` and the v8/v9/v10 parity sweeps).
* "cortiq-engine 0.8.43, src/gpu_wgpu/train_mm.rs" -- the ``blr`` layer
  (module doc, ``expand`` kernels, ``blr_forward``, ``blr_backward`` and the
  f64 host reference of test ``blr_layer_matches_host``).

Parity status: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py`` (closed forms, one-hot blocks, bit positions,
finite differences, library special cases).  No function is unpinned.
"""
from . import blr, f16, tq2  # noqa: F401
