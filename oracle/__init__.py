"""float64 CPU oracle for Grouped Cross-Attention with causal chunk retrieval.

Test infrastructure only: the tests, the package smoke check and the benchmark's CPU
baseline may import it; the library never does.
"""
from .gca_oracle import *  # noqa: F401,F403
