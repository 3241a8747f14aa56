"""fp64 CPU oracle (test infrastructure only; never imported by the library).

Only tests/, __graft_entry__.smoke() and bench.py's oracle legs import it.
"""
