"""CPU oracle for the SVDQuant W4A4 (NVFP4 / E2M1) linear layer.

TEST INFRASTRUCTURE ONLY.  The oracle is a plain, slow restatement of the
method on the host (numpy; float64 for products, float32 IEEE operations where
the encoding fixes float32).  Only the test-suite, the smoke check of the
package's graft entry and the CPU baseline leg of the benchmark may import it.
The CUDA library never calls it and shares no code with it.

Modules:
  nvfp4     -- E2M1 / E4M3 encodings and the 16-element block quantiser
  int4      -- the INT4 variant's 64-element group quantiser
  svdquant  -- smoothing, low-rank split, residual quantisation, forward pass

Parity status of each function is listed in the module headers.
"""
from . import int4, nvfp4, svdquant  # noqa: F401
