"""The build entry point compiles (or finds up to date) both shared libraries and checks
that the loaded library matches the declared header version."""

import __graft_entry__ as entry


def test_build_entry_point():
    entry.build()
