"""GPU: the debug build of the library (liboscar_debug.so: the same kernels compiled with OSCAR_DEBUG, whose
device-side bounds checks of workspace, partial-slot and pool indices set OSCAR_DEVERR_DEBUG_CHECK and skip the
access instead of trapping) gives the oracle's results with no check failing.  It runs in a child process that
sets OSCAR_DEBUG=1, so that the binding loads the debug library there."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import numpy as np, torch
import bit_rotated_kv_02_gb300 as ok
import synth
from tests import helpers
assert ok.lib()._name.endswith("liboscar_debug.so"), ok.lib()._name
for (lens, Hq, Hkv, g, seed) in (([330, 1100], 8, 2, 128, 31), ([5, 320, 900] + [400] * 30, 32, 8, 128, 32),
                                 ([700, 1500], 16, 2, 32, 33)):
    B = len(lens)
    pages = [max(0, -(-(L - 320 + 4) // 64)) for L in lens]
    O, P = helpers.make_pools(B, Hq, Hkv, g, pages, seed)
    ch = synth.outlier_channels(seed, Hkv, 128, 4)
    for b, L in enumerate(lens):
        K = synth.outlier_kv(seed + 10 + b, L, Hkv, 128, ch)
        V = synth.outlier_kv(seed + 500 + b, L, Hkv, 128, ch)
        O.prefill(b, K, V)
        ok.oscar_prefill_pool(P, b, helpers.to_dev_bf16(K), helpers.to_dev_bf16(V))
    q = synth.outlier_q(seed + 7, B, Hq, Hkv, 128, ch)
    out = ok.oscar_decode_attention(P, helpers.to_dev_bf16(q))
    helpers.assert_attention_close(out.cpu().numpy(), O.decode(q))
    for t in range(3):
        kn = synth.outlier_kv(seed + 2000 + t, B, Hkv, 128, ch)
        vn = synth.outlier_kv(seed + 3000 + t, B, Hkv, 128, ch)
        O.append(kn, vn)
        out = ok.oscar_decode_step(P, helpers.to_dev_bf16(kn), helpers.to_dev_bf16(vn), helpers.to_dev_bf16(q))
        helpers.assert_attention_close(out.cpu().numpy(), O.decode(q))
    torch.cuda.synchronize()
    helpers.assert_pools_equal(O, P)
    assert P.err() == 0, hex(P.err())
print("debug build ok:", ok.lib()._name)
"""


def test_debug_build_runs_clean_and_matches_the_oracle():
    from bit_rotated_kv_02_gb300 import build
    build.build(debug=True)
    env = dict(os.environ, OSCAR_DEBUG="1", PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "debug build ok" in r.stdout and "liboscar_debug.so" in r.stdout
