"""okv: lookahead sparse KV staging and sparse decode attention on one GB300 (sm_103a).

The compute path is the CUDA library ``libokv.so`` (C ABI in ``include/okv.h``); this
package is its Python binding (argument marshalling only). There is no CPU fallback: if the
library is missing, :func:`load_library` (called by every :class:`Context`) raises ImportError.
"""
from .binding import (BF16, F32, Config, Context, HostBuffer, OkvError, library_path,  # noqa: F401
                      load_library)
