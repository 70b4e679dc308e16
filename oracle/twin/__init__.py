"""A second, independent writing of the oracle's definitions in numpy (float64).

Test infrastructure only: ``tests/test_oracle_twin.py`` checks the C++ oracle against it on small
cases, so that a slip in either writing shows as a disagreement.  Nothing else uses it.
"""
from . import head, layers, lut6, model, quantize  # noqa: F401
