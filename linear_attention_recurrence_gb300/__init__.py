"""GB300-native Gated DeltaNet prefill recurrence.

* ``gdn``    - the Python binding of libgdn.so (gdn_recurrence, gdn_out_norm, ...).
* ``inputs`` - seeded synthetic inputs of the prefill shapes.
* ``build``  - nvcc build of libgdn.so for sm_103a.
"""
from . import inputs  # noqa: F401
from .gdn import (GDN_AUTO, GDN_CHUNKED, GDN_SEQUENTIAL, GDNError, gdn_chunked_scratch_bytes,  # noqa: F401
                  gdn_decode, gdn_device_status, gdn_last_error, gdn_launch_count, gdn_out_norm, gdn_recurrence,
                  gdn_poison_scratch, gdn_release_scratch, load_library)
