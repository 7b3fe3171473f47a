"""CPU float64 oracle (test infrastructure only; see ssb_oracle.py)."""
from . import ssb_oracle  # noqa: F401
