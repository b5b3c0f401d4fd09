"""Per-case parity errors of the GPU tests, kept for the session and written out at its end.

Every call of ``gpu_path.assert_close`` adds one record (test id, case, output dtype, max abs error,
max relative error over |ref| >= 0.1, the tolerance it was held to).  With PKV_PARITY_LOG set to a
file path, the session writes the records there as JSON (``conftest.pytest_sessionfinish``), so the
measured errors of a GPU run can be kept beside its pass count.
"""
RECORDS = []
