"""CPU oracle of the KV-cache compression path (test infrastructure only)."""
