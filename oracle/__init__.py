"""CPU oracle for the prefix-cached flow-matching action expert (test infrastructure only)."""
from .vla_oracle import *  # noqa: F401,F403
from .vla_oracle import __all__  # noqa: F401
