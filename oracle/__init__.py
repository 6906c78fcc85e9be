"""fp64 CPU oracle for the attention hot path.  Test infrastructure only: the
product path never imports it (see oracle/attention.py)."""
from .attention import *  # noqa: F401,F403
