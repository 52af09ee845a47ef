"""B300-native multiresolution hash-grid encoding (Hermite-NGP and d-linear
Instant-NGP) -- Python side of the C-ABI library ``libhg.so``.

``from multiresolution_hash_grid_02_b300 import hg`` gives the binding with the
C entry-point names (``hg.hg_encode_fwd`` ...); ``workloads`` holds the
seeded synthetic inputs.  Importing the
package does not load the CUDA library; the first call does, and raises if it
is missing.
"""
from . import _binding as hg  # noqa: F401
from ._binding import (GridDesc, SirenDesc, TableView, HGError, packed_views, order_views, linear_view,  # noqa: F401
                       HG_F32, HG_F16, HG_POINT_MAJOR, HG_FEATURE_MAJOR)
