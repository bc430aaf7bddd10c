"""CPU oracle (test infrastructure only; see qsa_oracle's header)."""
from . import qsa_oracle  # noqa: F401
