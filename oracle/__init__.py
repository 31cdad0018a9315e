"""fp64 CPU oracle for the PISA hot path -- test infrastructure only (see pisa_oracle)."""
