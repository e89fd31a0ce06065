"""Two host threads, each with its own problem (one forcing the generic
kernels, one the tcgen05 kernels) and its own stream, call
moe_fused_experts at the same time.  The kernel family is a field of each
problem, and with stage timing off no call takes a process-wide lock, so the
threads neither serialise nor see each other's choice: both outputs match the
oracle."""
import threading

import pytest
import torch

from helpers import compare, run_oracle, to_device
from moe_workloads import make_custom, to_host

pytestmark = pytest.mark.gpu


def test_two_threads_two_streams_two_paths():
    import quantized_moe_expert_topk_gb300 as moe
    wl = make_custom(M=300, K=256, N=192, E=4, T=2, wfmt="fp8_block128", afmt="fp8_group128_dyn",
                     seed=31, name="threads")
    ref = run_oracle(wl, None, to_host(wl))
    wl = to_device(wl)
    outs, errors = {}, []

    def worker(path):
        try:
            layer = moe.FusedExperts.from_workload(wl, path=path)
            s = torch.cuda.Stream()
            out = torch.empty((wl.M, wl.K), dtype=torch.bfloat16, device="cuda")
            with torch.cuda.stream(s):
                for _ in range(20):
                    layer(wl.x, wl.topk_ids, wl.topk_weights, wl.expert_map, out=out, stream=s)
            s.synchronize()
            outs[path] = out
        except Exception as e:  # reported by the main thread
            errors.append((path, e))

    threads = [threading.Thread(target=worker, args=(p,)) for p in ("generic", "tc")]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for path, out in outs.items():
        err, tol, rms = compare(wl, out, ref)
        assert rms > 0 and err <= tol, (path, err, tol)
    assert moe.moe_get_device_error() == 0
