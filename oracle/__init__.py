"""fp64 CPU oracle for the Llama-architecture single-token decode step.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.  Only the test suite, the
package smoke check and the benchmark's CPU-baseline leg may import this
package.  It shares no code with the CUDA library (no kernels, headers,
tables or helpers); both read the same quantised weight bytes, produced by the
separate ``synth`` input generator.

It is the plain definition of what the decode step computes, written out in
NumPy float64 with no blocking, fusion or reordering beyond what the
definition states:

* ``quant``  - Q8_0 / Q4_0 block dequantisation.
* ``ops``    - RMSNorm, RoPE, causal GQA attention with softmax, SiLU/SwiGLU,
               fp16 rounding of the KV cache.
* ``model``  - embedding, the per-layer decode step, final norm, LM head,
               greedy pick, prefill, the KV fork, layer skip and
               self-speculative decoding.
* ``kquant`` - Q4_K / Q6_K super-block dequantisation and the dequant-GEMV.

Sources (by page and section): the pure C + CUDA inference engine page (rskf.cn),
section 1 (the engine implements RoPE, GQA, SwiGLU, RMSNorm and a KV cache for
the Llama architecture, and covers the Q4_0 and Q8_0 formats) and section 4.4
(custom CUDA operators: single-token GEMV, fused RMSNorm, RoPE with a
precomputed sin/cos table, SwiGLU fused with the projection, causal softmax
with the mask inside); the SwarmKV page ("Prefill once, fan out"), section 2
(prefill fills the per-layer KV cache, decode extends it token by token) and
sections 3-4 (the forked branches continue RoPE positions at the prefix
length).  The pages give no formulas; the readings taken where they are
silent are listed in each function's docstring.

Parity status: every op is pinned by tests against closed forms, invariants
or brute force (the K-quant formats by blocks written field by field from the
stated layout, and by planted mistakes that the pins must catch).  The composed model is pinned by self-consistency (prefill of
T tokens equals T decode steps; a fork equals an independent prefill) and by
wiring cases with closed forms; there is no external worked example, so the
full-model composition beyond those is "parity unpinned".
"""
from . import quant, ops, model, kquant  # noqa: F401
from .model import OracleModel, OracleSeq  # noqa: F401
