"""CPU oracle for the fused MoE layer (forward + backward).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of the package entry
file and the `cpu_baseline` / reference leg of the benchmark may import this
package.  The CUDA library never calls it, links it or falls back to it, and it
shares no code with the CUDA path: the one shared module is the seeded input
generator, which holds none of the layer's arithmetic.

Source pages: "Prime Intellect releases Prime Mega MoE" (English article,
sections "Why is MoE training communication-bound?" and "How does the fused
kernel work?"; the Russian rewrite on the-ai.news, section "Объединённое ядро,
дополненное для обучения").  They name the steps -- tokens sorted by expert,
dispatched, the two expert linear layers with SwiGLU between them, combined
back, and a backward pass -- and the BF16 / MXFP8 / fp8_bwd precisions.  They
give no formulas; every formula here is the plainest mathematical reading of
those steps, listed in the repository's design notes.

Parity status: every function here is pinned by tests that do not reuse its own
formulas (brute-force routing, the dense SwiGLU MLP of torch.nn.functional for
k=1, identical-expert and linearity invariants, central finite differences for
every gradient, torch's float8_e4m3fn rounding for the MXFP8 element grid).
"""
from .moe import (route, forward, backward, expert_forward, expert_backward,  # noqa: F401
                  sigmoid, silu, swiglu, swiglu_grad, PRECISIONS)
from .mx import mx_qdq, e4m3_round, e8m0_scale_exponent  # noqa: F401
