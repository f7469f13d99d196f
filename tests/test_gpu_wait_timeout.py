"""The decode's abort path, made to run on purpose in a test build of the library.

Every wait inside the decode kernel on another role's progress is bounded; when one runs
out the CTA raises its abort flag, every role leaves its loop at its next wait, the CTA
lets its own copies and MMAs in flight land, frees its tensor memory, meets its cluster
peer at the final barrier and reports MLA_STATUS_WAIT_TIMEOUT in the status word.  The
fault-injection build (same sources, waits limited to 20 ms) makes CTA 0 leave one tile
of its schedule unloaded, so that the waits on that tile run out: nothing faults, traps or
hangs, the call returns, the status word carries the timeout bit, and the next calls on
the same GPU -- through the test build and through the shipped library -- are clean and
match the oracle.  It runs in a child process of its own."""
import json
import os
import subprocess
import sys

import pytest

from mla_latent_kv_split_gb300 import binding as mb
from mla_latent_kv_split_gb300 import build

HERE = os.path.dirname(os.path.abspath(__file__))


def test_shipped_library_has_no_fault_injection():
    if not os.path.exists(mb.LIB_PATH):
        build.build()
    assert not hasattr(mb.lib(), "mla_fault_injection_drop_tile")
    assert os.path.basename(mb.LIB_PATH) == "libmla_decode.so" != os.path.basename(build.FAULT_LIB)


@pytest.mark.gpu
def test_wait_timeout_aborts_cleanly_and_the_next_call_is_clean():
    r = subprocess.run([sys.executable, os.path.join(HERE, "_wait_timeout_child.py")], capture_output=True, text=True,
                       timeout=600)
    lines = [l for l in r.stdout.splitlines() if l.startswith("RESULT ")]
    assert r.returncode == 0 and lines, f"child failed ({r.returncode}):\n{r.stdout[-3000:]}\n{r.stderr[-3000:]}"
    res = json.loads(lines[-1][len("RESULT "):])
    print(res)
    assert res["dropped_rc"] == 0
    assert res["dropped_status"] & 0x10, hex(res["dropped_status"])
    assert res["dropped_seconds"] < 5.0
    assert res["next_rc"] == 0 and res["next_status"] == 0, res
    assert res["next_matches_oracle"] is True, res["next_matches_oracle"]
    assert res["shipped_status"] == 0 and res["shipped_matches_oracle"] is True, res
