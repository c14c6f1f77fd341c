"""CPU oracle: test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  It shares no code with the CUDA
library and the library never imports it.
"""

from . import kvq_oracle, layout  # noqa: F401
