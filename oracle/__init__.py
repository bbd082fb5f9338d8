"""CPU oracle for the tiered KV-cache decode path (test infrastructure only).

Imported by the tests, by ``__graft_entry__.smoke`` and by the benchmark's CPU
baseline leg. The library never imports it.
"""
from .qevict_oracle import *  # noqa: F401,F403
