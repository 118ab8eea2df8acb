"""Coverage-selected sparse decode over a paged KV cache, for GB300 (sm_103a).

The compute path is libasp.so (CUDA kernels behind a C ABI, include/asp.h);
`binding` marshals torch tensors into it, `step` strings the calls of one
decode step together (and captures them into a CUDA graph), and `synth`
draws seeded synthetic workloads. Importing the package loads nothing; the
library is loaded on first use and its absence is an error.
"""

__all__ = ["binding", "step", "synth", "build"]
