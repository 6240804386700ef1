"""First calls of moe_w2_forward from several host threads at once.

The library sets kernel attributes and reads occupancy once per device on the
first call of each path; those set-ups are serialised inside the library, and
the ctypes binding releases the GIL, so several threads really enter it
together.  The check runs in a fresh process (so that the calls are the
first ones) with one thread per kernel path (mma.sync decode, block-scaled
decode, prefill) on its own stream, and compares every output bit for bit with
a later sequential run of the same calls.
"""
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

_CHILD = textwrap.dedent(
    """
    import threading
    import numpy as np
    import torch
    from bit_moe_expert_w2_gb300 import inputs, moe_w2

    # (H, I, E, k, T, seed): with the stream-K kernel selected, 2 pairs and 6
    # pairs take it, 32 pairs the block-scaled kernel, 160 pairs the prefill
    # kernels, and I = 256 the mma.sync decode kernel
    moe_w2.set_decode_stream(True)
    cases = [(512, 512, 8, 2, 1, 21), (512, 512, 8, 2, 16, 22), (512, 512, 8, 2, 80, 23), (512, 512, 8, 2, 3, 24),
             (512, 256, 8, 2, 3, 25)]
    args = []
    for c in cases:
        lay = inputs.small_layer_inputs(*c)
        planes = {n: torch.from_numpy(np.ascontiguousarray(v)).cuda() for n, v in lay.planes.items()}
        x = torch.from_numpy(np.ascontiguousarray(lay.x).view(np.int16)).cuda().view(torch.bfloat16)
        args.append((x, torch.from_numpy(lay.ids).cuda(), torch.from_numpy(lay.weights).cuda(), planes))
    torch.cuda.synchronize()

    outs = [None] * len(args)
    errs = []
    go = threading.Barrier(len(args))

    def work(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                st = torch.zeros(1, dtype=torch.int32, device="cuda")
                go.wait()
                y = moe_w2.forward(*args[i], status=st, stream=s)
                s.synchronize()
                outs[i] = (y.view(torch.int16).cpu().numpy(), int(st.item()))
        except BaseException as e:
            errs.append(repr(e))

    th = [threading.Thread(target=work, args=(i,)) for i in range(len(args))]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert not errs, errs
    for i, a in enumerate(args):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        y = moe_w2.forward(*a, status=st)
        ref = y.view(torch.int16).cpu().numpy()
        assert outs[i][1] == 0 and int(st.item()) == 0, (i, outs[i][1], int(st.item()))
        assert np.array_equal(outs[i][0], ref), f"case {cases[i]}: threaded output differs from the sequential one"
    print("ok")
    """
)


def test_first_calls_from_concurrent_threads_match_sequential_calls():
    r = subprocess.run([sys.executable, "-c", _CHILD], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert r.stdout.strip().endswith("ok")
