"""CPU oracle for the selective scan (test infrastructure only; see oracle.py)."""
