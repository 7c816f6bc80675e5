"""CPU oracle for the work-decomposed BF16 GEMM.

TEST INFRASTRUCTURE, not part of the library. Only the tests, the package's
smoke check and the benchmark's CPU-baseline / reference arm may import it.
It shares no code with the CUDA path and imports nothing from it; the two
meet only in the seeded inputs of the top-level `synth` module.

- `oracle.schedule`: wave arithmetic, the data-parallel, Split-K, Stream-K and
  hybrid decompositions as an integer work-unit map, the fixup ownership rule,
  and the makespan cost model.
- `oracle.gemm`: the FP64 dot-product GEMM over the BF16-rounded inputs, and
  the per-split FP64 partial slabs.

Sources (all on the page "Split-K and Stream-K: The Last Wave of a GEMM",
kanthi.in, unless stated): the Mental model figure (toy 4-SM case), Case 1
(wave arithmetic), Case 2 (cost model, cutlass_heuristic, hybrid), Case 3
(k-order fixup, FP64 reference), Case 4 (reduction modes, max_sk_groups_); the
"Consecutive-B split-K NAX GEMM" report (docs.waffuru.ai), section "Contract
and numerical coverage" (NT layout, [splits,M,N] partials, FP64 dot products
over the rounded inputs); and the CUTLASS "Optimization Techniques" page
(Split-K factor heuristic, tile rasterization).
"""
