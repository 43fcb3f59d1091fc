"""fp64 CPU oracle of the compression step: test infrastructure only (see tri_oracle)."""
