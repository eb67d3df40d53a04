import pathlib
import sys

ROOT = pathlib.Path(__file__).resolve().parent.parent
for p in (str(ROOT), str(ROOT / "tests")):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device and the built library")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def oracle_rows():
    """The oracle over row ranges on every host core (full-size parity)."""
    from oracle_rows import OracleRows
    pool = OracleRows()
    yield pool
    pool.close()
