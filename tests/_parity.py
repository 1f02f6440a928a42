"""Error bookkeeping for the GPU parity tests.

``err`` returns the normwise relative error ``max|gpu - ref| / max|ref|``,
the figure the tolerances bound, and records it together with the
element-wise diagnostic ``max_i |gpu_i - ref_i| / max(|ref_i|, 1e-6 max|ref|)``
under the running test's id; ``tests/conftest.py`` prints the table at the
end of the session."""
import os

import oracle as O

RECORDS = []


def err(gpu, ref, what: str = "") -> float:
    n = O.relerr(gpu, ref)
    e = O.relerr_elementwise(gpu, ref)
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    RECORDS.append((test, what, n, e))
    return n
