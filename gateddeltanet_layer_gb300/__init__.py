"""GatedDeltaNet layer on GB300 (placeholder; binding added with the C-ABI)."""
