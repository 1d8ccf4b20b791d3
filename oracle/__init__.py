"""Float64 CPU oracle for the quantized-KV attention path.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's CPU
baseline leg are the only callers.  The CUDA library does not import, link or
run anything here, and nothing here imports the library.
"""
from .kvq_oracle import *  # noqa: F401,F403
