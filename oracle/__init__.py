"""CPU fp64 oracle for the compressed-KV decode path (test infrastructure only)."""
