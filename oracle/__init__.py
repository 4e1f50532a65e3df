"""CPU oracle of the HiSparse top-k sparse decode path (test infrastructure
only: used by tests/, __graft_entry__.smoke() and bench.py's CPU legs)."""
