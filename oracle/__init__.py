"""fp64 CPU oracle for exact attention.  Test infrastructure only (see oracle.py)."""
