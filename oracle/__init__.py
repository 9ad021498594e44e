"""CPU oracle (test infrastructure only; see ``oracle.moe_oracle``)."""
from .moe_oracle import *  # noqa: F401,F403
from . import moe_oracle  # noqa: F401
