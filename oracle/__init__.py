"""CPU float64 oracle (test infrastructure only; see ``oomb_oracle``).

Importable only from ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs
of ``bench.py``.  The product path never imports it.
"""
from .oomb_oracle import *  # noqa: F401,F403
from .oomb_oracle import __all__  # noqa: F401
