"""CPU oracle (test infrastructure only): see ``oracle.tq_oracle``."""
from .tq_oracle import *  # noqa: F401,F403
from .tq_oracle import __doc__  # noqa: F401
