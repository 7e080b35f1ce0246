import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libmala.so")
    config.addinivalue_line("markers", "slow: long-running CPU oracle cases")


def pytest_terminal_summary(terminalreporter):
    """One line on how often the parity checks met a borderline tile that the
    GPU decided the other way (and so compared against the oracle's replay)."""
    parity = sys.modules.get("tests.parity")
    if parity is None:
        return
    st = parity.REPLAY_STATS
    if st["fwd_blocks"] or st["decode_rows"] or st["bwd_tiles"]:
        terminalreporter.write_line(
            "parity replays: forward {fwd_replayed} of {fwd_blocks} query blocks, decode {decode_replayed} of "
            "{decode_rows} rows, backward {bwd_replayed_tiles} of {bwd_tiles} tiles; borderline tiles taken the "
            "other way {overridden_tiles}".format(**st))
