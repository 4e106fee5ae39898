"""CPU oracle of the budgeted KV-cache compaction pass (test infrastructure only).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The library and its binding never import it.
"""
from .kvc_oracle import *  # noqa: F401,F403
from . import kvc_oracle  # noqa: F401
