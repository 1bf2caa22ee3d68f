import pytest


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (a B300, sm_103a)")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()
