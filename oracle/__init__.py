"""FP64 CPU oracle (test infrastructure only; see ``oracle.model``)."""
from . import model  # noqa: F401
