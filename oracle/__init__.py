"""fp64 CPU oracle of the vision-tower front end (test infrastructure only).

Only tests, the smoke check and the benchmark's CPU-baseline leg import this
package; the product path never does.
"""
from .oracle import *  # noqa: F401,F403
