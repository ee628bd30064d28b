"""Failure detection on the GPU without a fault.

Every wait of the tcgen05 kernels is bounded (2 s); when one runs out the
kernel records `stage | DSA_DEVERR_TIMEOUT` in the device error word, its roles
leave their loops, TMEM is freed and the kernel returns. Here the wait is made
to run out on purpose: with DSA_TEST_DROP_ARRIVE set, the tensor-core forward
skips one producer arrive in its first CTA, so the issuer's wait on that stage
never completes. The run happens in a child process (the switch is read once
per process). The test checks the reported status and that the context still
computes correct results afterwards.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent(f"""
    import sys
    sys.path.insert(0, {ROOT!r})
    sys.path.insert(0, {os.path.join(ROOT, "tests")!r})
    import numpy as np
    import torch
    import sparse_attention_index_gb300 as dsa
    import oracle
    import synth
    from gpu_util import TOL, bf16_dev, dev, host_f64, rel_err

    # tensor-core forward shape: 128 heads, Dqk 192, Dv 128
    B, S, H, k = 1, 300, 128, 64
    wl = synth.Workload("failure", seed=11, B=B, S=S, Hi=4, Di=32, topk=k, H=H, Dqk=192,
                        Dv=128, backward=False)
    att = synth.attention_inputs(wl)
    idx = np.full((B, S, k), -1, dtype=np.int32)
    for t in range(S):
        m = min(k, t + 1)
        idx[0, t, :m] = np.arange(t + 1 - m, t + 1)
    O, lse = dsa.dsa_sparse_attn_fwd(bf16_dev(att["Q"]), bf16_dev(att["K"]), bf16_dev(att["V"]),
                                     dev(idx), wl.scale)
    code = dsa.dsa_get_last_device_error()
    print("CODE", code)

    # the context still works: the indexer and the top-k on a small case, exact
    ind = synth.indexer_inputs(synth.WORKLOADS["tiny_s128"])
    sc = dsa.dsa_index_scores(bf16_dev(ind["q_idx"]), bf16_dev(ind["k_idx"]), dev(ind["w"]))
    ti, tc = dsa.dsa_topk(sc, 4)
    torch.cuda.synchronize()
    ref = oracle.index_scores(ind["q_idx"], ind["k_idx"], ind["w"], None)
    g = host_f64(sc[:, :, :128]).reshape(128, 128)
    ok_sc = all(np.array_equal(g[t, :t + 1], ref.reshape(128, 128)[t, :t + 1]) for t in range(128))
    ref_idx, _ = oracle.topk(ref.reshape(128, 128), None, 128, 4)
    ok_tk = np.array_equal(ti.cpu().numpy().reshape(128, 4), ref_idx)
    print("AFTER", int(ok_sc), int(ok_tk), dsa.dsa_get_last_device_error())
""")


def test_bounded_wait_timeout_is_reported_and_context_survives():
    env = dict(os.environ, DSA_TEST_DROP_ARRIVE="1")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=180)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = dict(l.split(" ", 1) for l in r.stdout.strip().splitlines() if " " in l)
    import sparse_attention_index_gb300 as dsa
    assert int(lines["CODE"]) == (dsa.DSA_STAGE_FWD | dsa.DSA_DEVERR_TIMEOUT)
    assert lines["AFTER"].split() == ["1", "1", "0"]
