"""The package entry point's smoke check, as the full test run calls it: one
tiny layer through each expert path the automatic choice takes, against the
oracle."""
import pytest

pytestmark = pytest.mark.gpu


def test_entry_point_smoke():
    import __graft_entry__
    __graft_entry__.smoke()
