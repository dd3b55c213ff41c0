"""CPU oracle for the ECHO decode hot path: test infrastructure only (see echo_oracle)."""
from .echo_oracle import *  # noqa: F401,F403
