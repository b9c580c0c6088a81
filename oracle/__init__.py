"""fp64 CPU oracle for batched draft-token verification (test infrastructure only;
see oracle/oracle.py's header for who may import it)."""
