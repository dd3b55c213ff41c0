"""ECHO decode hot path for one GB300: Python binding of the C-ABI library."""
