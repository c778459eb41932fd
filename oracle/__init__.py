"""CPU oracle for MTP speculative decoding: the draft block chained k times and
the verification of the drafted tokens.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links
this package: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA library; both sides
receive their inputs from the seeded generators, which hold none of the
method's arithmetic.

Everything here is plain numpy in float64, written step by step in the order
the pages give, with a library matmul as the only borrowed primitive:

* ``numerics``  -- exact bf16 widening and round-to-nearest-even bf16 rounding;
* ``block``     -- one application of the MTP module and the k-deep draft chain
                   ("The Tiny Draft Model Hidden Inside Qwen", sections "One step
                   deeper than the main model" and "What vLLM and SGLang do with
                   the weights"; "Optimize vLLM speculative decoding with FastMTP
                   heads", section "Why fine-tune a single MTP head");
* ``verify``    -- greedy longest-prefix acceptance, stochastic rejection
                   sampling with residual resample, and the bonus token ("The
                   Tiny Draft Model Hidden Inside Qwen", section "How the draft
                   becomes real output"; "Speculative Decoding and MTP: Why
                   Guessing Is Free", sections "Speculative decoding: draft, then
                   verify" and "It's exact, not approximate").

Parity status of each function is stated in its docstring.  The draft block's
numerics have no worked example on the pages: beyond the structural pins in the
tests (special cases, invariants, an independent loop evaluation) its GPU
comparison is "parity unpinned" up to the stated tolerance.
"""

from . import numerics, block, verify  # noqa: F401
