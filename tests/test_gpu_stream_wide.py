"""GPU parity of the fused streaming grid with 32-token passes (taken when the
local experts hold more than 32, and at most 64, slots each on average): MXFP4
w4a16 against the oracle, with experts of one to several passes, an empty
expert and both gate layouts."""
import zlib

import pytest

from helpers import compare, run_gpu, run_oracle, sample_tokens, to_device
from moe_workloads import make_custom, to_host

pytestmark = pytest.mark.gpu

CASES = [
    # name, M, K, N, E, T, gate
    ("wide_interleaved", 200, 256, 192, 8, 2, "interleaved"),   # 50 slots per expert
    ("wide_separated", 130, 320, 128, 8, 3, "separated"),       # 49 slots per expert
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_wide_passes_match_oracle(case):
    name, M, K, N, E, T, gate = case
    wl = make_custom(M=M, K=K, N=N, E=E, T=T, wfmt="mxfp4", afmt="bf16", act="swiglu_oai",
                     gate=gate, bias=True, seed=zlib.crc32(name.encode()) % 997,
                     name=f"stream/{name}")
    ids = wl.topk_ids
    ids[ids == 1] = 0  # expert 1 empty, expert 0 large (several passes)
    host = to_host(wl)
    ref = run_oracle(wl, None, host)
    out = run_gpu(to_device(wl), "stream")
    err, tol, rms = compare(wl, out, ref)
    assert err <= tol, f"{wl.name}: max|err| {err:.4e} > tol {tol:.4e} (rms {rms:.4e})"
