"""Shared pytest configuration: the ``gpu`` marker, and building the CUDA
library and the CPU oracle before any test module imports them (so a missing
build fails loudly instead of skipping)."""
import pytest


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")


def pytest_sessionstart(session):
    import __graft_entry__

    __graft_entry__._builder().build()
    import oracle

    oracle.build()


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    oracle.build()
    return oracle
