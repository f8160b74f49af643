"""CPU oracle for hybrid-precision (INT4 + BF16) attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
or run anything in this package.  The product path (the CUDA library and its
Python binding) never calls it and shares no code with it; the only shared
module is the seeded input generator ``gen``.

It is a plain, slow, obviously-correct restatement of what the method in
*HyQuant: Hybrid-Precision Quantization for LLM Attention* computes, in
float64; integer decisions (codes) are taken exactly, by their definition
(the nearest grid point, ties to even).  Each function names the passage it
follows.  It exists twice, written independently: the Python modules below
and ``cpp/hyq_oracle.cpp`` (plain C++17, float64 accumulation, its own
binary16 / e4m3 arithmetic; ``cpp_oracle`` binds it), and the tests assert
that the two agree.

Modules
-------
quant      asymmetric group quantiser Quant_B(.; G) and DeQuant (Alg. 4, Eq. 9)
select     vertical-line token identification (Eq. 4-5, Alg. 1)
attention  hybrid decode attention (Eq. 8-9, Alg. 3) and textbook softmax
prefill    hybrid prefill operator (Eq. 6-7, Alg. 2)
metrics    attention-output MSE and attention-mass coverage (Table 1, Fig. 2/6)
accounting byte counts of the hybrid cache (Table 14, §5.5)
cpp_oracle ctypes binding of the C++ restatement (quantiser, selection, decode,
           prefill), built by ``cpp_oracle.build()`` with g++

Pins: every function here is checked by ``tests/test_oracle_*.py`` against
closed forms, special cases that reduce to a library routine, brute force on
tiny inputs and invariants.  Functions without such a pin say
"parity unpinned" in their docstring.
"""
