"""fp64 / fp32 CPU oracle for Gram Newton-Schulz and the Muon step.

TEST INFRASTRUCTURE ONLY: tests/, __graft_entry__.smoke() and bench.py's CPU
legs import it; the library never does. See gram_ns.py and muon.py for what
each function follows on the pages.
"""
from . import gram_ns, muon  # noqa: F401
