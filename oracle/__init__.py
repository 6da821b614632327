"""CPU oracle for the Mixture-of-Kittens MoE layer.

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, float64 NumPy
statement of what the layer computes.  It exists to check the CUDA library
and nothing else: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import it.  The library and its
Python binding never import it, and the two share no code (no kernels, no
headers, no helpers, no constants); only the seeded input generators in
``mixture_experts_layer_side_gb300.inputs`` feed both sides.

Modules
-------
``moe``        schedule, forward and backward of the routed SwiGLU MoE layer
``mxfp8``      E4M3 / E8M0 block quantisation (32-element blocks)
``heuristics`` the two-wave minibatch floor
``router``     top-k softmax router: selection, scores, logit and weight gradients

Parity status (what pins each function, see ``tests/test_oracle.py``):

* ``moe.build_schedule``  -- brute-force sort on tiny inputs, invariants.
* ``moe.forward``         -- brute-force dense routing, dense-MLP special case,
                             token-permutation invariance, W2 = 0.
* ``moe.backward``        -- float64 autograd of the dense formulation,
                             central finite differences, permutation
                             invariance, empty experts.
* ``mxfp8``               -- exhaustive nearest-code search over all 256 E4M3
                             codes, exact round trips, power-of-two scales.
* ``moe`` in MXFP8 mode   -- forward and backward against the layer written
                             per routed row with an exhaustive-search
                             quantiser at every quantisation point (per-expert
                             row blocks for the weight gradients), and
                             identity on pre-quantised data.
* ``heuristics``          -- the 2,368-token floor printed for the Kimi-2.5
                             shape (golden fixture).
* ``router``              -- brute-force selection with ties, softmax special
                             cases, float64 autograd, finite differences, and
                             the layer's score gradient composed with the
                             router backward against autograd of the whole
                             routed network (``tests/test_oracle_router.py``).
"""

from . import heuristics, moe, mxfp8, router  # noqa: F401
