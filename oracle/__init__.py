"""CPU oracle of Invariant Bit Packing: test infrastructure only.

``ibp_ref`` is a pure-Python bit-by-bit reference with the word width as a
parameter; ``oracle_c`` wraps an independent bit-by-bit C reference for
table-sized inputs.  The product library never imports this package.
"""
