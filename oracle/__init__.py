"""CPU oracle for the budgeted KV-compression + ragged-decode path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
anything in this package.  The product path (the C-ABI library and its Python
binding) never imports it, and this package imports nothing from the product.
"""
from .kvc_oracle import *  # noqa: F401,F403
