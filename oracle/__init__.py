"""fp64 CPU oracle of the grouped-query attention block (test infrastructure only)."""
