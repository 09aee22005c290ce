"""CPU oracle of the Medusa decode step -- TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 restatement of what each step computes, written from the
method's pages and shared with nothing in the CUDA library.  Only the tests, the
smoke check and the bench's CPU-baseline leg may import it; the product path
never does.

Modules:
  oracle.oracle    ctypes wrapper of the C oracle (medusa_oracle.c)
  oracle.analytic  closed forms of the speculative-decoding cost model
"""
