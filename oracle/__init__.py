"""fp64 CPU oracle for two-stream BDLM attention (test infrastructure only;
see ``oracle.bdlm_oracle``)."""
from .bdlm_oracle import *  # noqa: F401,F403
