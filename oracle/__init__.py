"""fp64 CPU oracle for the MSA block-sparse attention backward (test infrastructure only)."""
