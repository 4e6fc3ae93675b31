"""fp64 CPU oracle for exact paged attention -- test infrastructure only.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
legs may import this package.  It shares no code with paged_kv_cache_03_gb300.
"""
from .oracle import (ORACLE_ERR_BAD_BLOCK_TABLE, ORACLE_ERR_INVALID_ARG, ORACLE_OK,  # noqa: F401
                     OracleError, OracleLib, build, host_cores, load)
