"""Several host threads calling the library at once.

The first decode or prefill call on a device raises its kernels' shared-memory limit;
several threads may reach that set-up together.  A fresh process (so that no earlier
call has done the set-up) starts four threads behind a barrier; each calls pa_decode and
pa_prefill_chunk on its own stream, at once.  Every call must succeed and every thread's
output must equal the serial result bit for bit (both kernels are deterministic).
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent(r"""
    import sys, threading
    import torch
    sys.path.insert(0, sys.argv[1])
    import workloads
    import paged_kv_attention_write_gb300 as pa

    def upload(case):
        t = {k: getattr(case, a).cuda() for k, a in
             [("q", "query"), ("kc", "key_cache"), ("vc", "value_cache"), ("bt", "block_tables"),
              ("cl", "context_lens"), ("qsl", "query_start_loc")]}
        pa.pa_reshape_and_cache(case.new_key.cuda(), case.new_value.cuda(), t["kc"], t["vc"],
                                case.slot_mapping.cuda())
        return t

    dec = workloads.make_decode_case("thr-d", [700, 3000, 64, 1500], 16, 32, 8, 128, torch.bfloat16, 3)
    pre = workloads.make_prefill_case("thr-p", [0, 300], [100, 257], 16, 32, 8, 128, torch.bfloat16, 4)
    td, tp = upload(dec), upload(pre)
    torch.cuda.synchronize()
    mq = int((pre.query_start_loc[1:] - pre.query_start_loc[:-1]).max())
    n = pa.pa_decode_workspace_size(dec.num_seqs, 32, 8, 128, dec.max_context_len)

    def run(results, i, barrier):
        try:
            stream = torch.cuda.Stream()
            ws = torch.empty(n, dtype=torch.uint8, device="cuda")
            od = torch.empty(tuple(dec.query.shape), dtype=torch.float32, device="cuda")
            op = torch.empty(tuple(pre.query.shape), dtype=torch.float32, device="cuda")
            torch.cuda.synchronize()
            barrier.wait()
            with torch.cuda.stream(stream):
                pa.pa_decode(od, td["q"], td["kc"], td["vc"], td["bt"], td["cl"], dec.max_context_len,
                             dec.scale, workspace=ws)
                pa.pa_prefill_chunk(op, tp["q"], tp["qsl"], mq, tp["kc"], tp["vc"], tp["bt"], tp["cl"],
                                    pre.max_context_len, pre.scale)
            stream.synchronize()
            results[i] = (od.cpu(), op.cpu())
        except Exception as e:  # reported by the main thread
            results[i] = e

    nthreads = 4
    results = [None] * nthreads
    barrier = threading.Barrier(nthreads)
    threads = [threading.Thread(target=run, args=(results, i, barrier)) for i in range(nthreads)]
    for t in threads: t.start()
    for t in threads: t.join()
    for r in results:
        if isinstance(r, Exception):
            raise r
    serial = [None]
    run(serial, 0, threading.Barrier(1))
    for od, op in results:
        assert torch.equal(od, serial[0][0]) and torch.equal(op, serial[0][1])
        assert torch.isfinite(od).all() and torch.isfinite(op).all()
    print("threads ok")
""")


def test_concurrent_first_calls_from_several_threads(cuda_ok):
    r = subprocess.run([sys.executable, "-c", SCRIPT, ROOT], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "threads ok" in r.stdout
