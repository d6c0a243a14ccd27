"""KDA decode / spec-verify core for GB300 (placeholder; binding follows)."""
