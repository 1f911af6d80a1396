"""CPU oracle for the MoE expert layer (test infrastructure).

`oracle.cpp` is the oracle: a plain C++17 + OpenMP definition of the layer in
double precision (moe_oracle.cpp) behind a ctypes binding.  `oracle.moe_oracle`
restates the same definition in float64 numpy and serves only as an
independent cross-check of the C++ one.  Nothing here is product code: only
the tests, the package smoke check and the benchmark's CPU-baseline leg use it.
"""
