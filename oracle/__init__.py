"""CPU oracle for the MuonClip step.  Test infrastructure only: imported by
tests/, the smoke check and the CPU-baseline leg of the benchmark, never by the
library's product path."""
from .muonclip_oracle import *  # noqa: F401,F403
