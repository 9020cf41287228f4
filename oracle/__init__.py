"""CPU oracle of the DSA step: test infrastructure, not part of the product.

Only the tests, the smoke check and the benchmark's CPU-baseline arm import
this package.
"""
from .dsa_oracle import *  # noqa: F401,F403
