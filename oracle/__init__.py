"""Plain CPU oracle for KDA (test infrastructure only; see oracle.py)."""
