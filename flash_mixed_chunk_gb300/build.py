"""Command line: ``python -m flash_mixed_chunk_gb300.build [--force] [-v]``
compiles libflash_mca.so in-tree for sm_103a (see ``_buildlib``)."""
import sys

from flash_mixed_chunk_gb300 import _buildlib

if __name__ == "__main__":
    print(_buildlib.build(force="--force" in sys.argv, verbose="-v" in sys.argv))
