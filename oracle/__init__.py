"""CPU oracle (test infrastructure only; see mq_oracle.py)."""
from .mq_oracle import *  # noqa: F401,F403
from . import mq_oracle  # noqa: F401
