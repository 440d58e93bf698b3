"""CPU oracle for the update phase of SS-HSDP (runtime/update-decoupled sharded
data parallelism): plain, slow, obviously-correct NumPy restatements of what
the update path computes.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check in the repo's
entry module and the benchmark's CPU-baseline / reference leg may import
anything from this package.  The product path (the C-ABI library and its
Python binding) never imports, calls or links it, and this package imports
nothing from the product: the two share no code.  The only module both sides
use is `workloads`, which holds input shapes and seeded draws and none of the
method's arithmetic.

Modules and what they follow (citations are to "SS-HSDP: Efficient and
Flexible Sharded Data Parallelism via Runtime-Update Decoupling"):
  views   - data tree (section 3.2 "Data Tree"), shard chain and fragments
            (section 3.2 "Shard Chain", "Distributed updates"), hierarchical
            rank order (section 4.2 "Fully Zero Copy", Figure 4), and the
            emulated rank-segment layout of one HBM allocation.
  muon    - f0 momentum, f1 Newton-Schulz, f2 main-weight update (section 3.1
            example EG1, section 3.4, Figure 4).
  adamw   - elementwise AdamW (section 2.3 / 5.2: AdamW updates the
            parameters Muon does not), PyTorch's documented algorithm.
  mxfp8   - G: MXFP8 quantization, E4M3 elements + UE8M0 scale per block
            (section 3.1 EG1, Figure 4; OCP Microscaling format, ref. [28]).
  update  - the composed update phase on logical arrays.

Every function here has a pin in tests/ against something other than itself;
see each module's docstring for its pins.
"""
