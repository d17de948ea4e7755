"""CPU oracle for the draft step. Test infrastructure only: see dflash_oracle.py."""
from .dflash_oracle import *  # noqa: F401,F403
