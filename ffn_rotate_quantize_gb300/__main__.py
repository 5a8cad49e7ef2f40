"""`python -m ffn_rotate_quantize_gb300`: the library's self-test on this machine (see selftest.py)."""
import sys

from .selftest import main

sys.exit(main())
