"""The C ABI's thread-safety claim: two host threads issue calls at the same
time, each on its own stream with its own inputs, and every result equals the
one a single thread gets, bit for bit.  Covers the device-pointer call and the
host-buffer call (whose enqueue is serialised per device)."""
import threading

import pytest

torch = pytest.importorskip("torch")

import gated_deltanet_chunked_gdr_gb300 as gdr  # noqa: E402
import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _inputs(seed, dev=None):
    wl = workloads.CONFIGS["B1_T8192_H8_K128"].with_(seed=seed)
    inp = workloads.make_inputs(wl)
    if dev is None:
        return {k: (None if v is None else v.pin_memory()) for k, v in inp.items()}
    return {k: (None if v is None else v.to(dev)) for k, v in inp.items()}


def _run_threads(work):
    errors = []

    def wrap(fn):
        try:
            fn()
        except Exception as e:          # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=wrap, args=(fn,)) for fn in work]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors


def test_device_calls_from_two_threads():
    dev = _dev()
    xs = [_inputs(71, dev), _inputs(72, dev)]
    refs = [gdr.kkt_solve(x["k"], x["g"], x["beta"], output_dtype=torch.bfloat16) for x in xs]
    torch.cuda.synchronize(dev)
    outs = [[None] * 20, [None] * 20]

    def worker(t):
        def fn():
            torch.cuda.set_device(dev)
            s = torch.cuda.Stream(dev)
            with torch.cuda.stream(s):
                for n in range(20):
                    outs[t][n] = gdr.kkt_solve(xs[t]["k"], xs[t]["g"], xs[t]["beta"],
                                               output_dtype=torch.bfloat16)
            s.synchronize()
        return fn

    _run_threads([worker(0), worker(1)])
    for t in range(2):
        for o in outs[t]:
            assert torch.equal(o, refs[t])
    assert gdr.device_status() == gdr.GDR_OK


def test_host_buffer_calls_from_two_threads():
    dev = _dev()
    xs = [_inputs(73), _inputs(74)]
    refs = []
    for x in xs:
        with torch.cuda.device(dev):
            r = gdr.kkt_solve_host(x["k"], x["g"], x["beta"], output_dtype=torch.float32)
        torch.cuda.synchronize(dev)
        refs.append(r.clone())
    outs = [[None] * 5, [None] * 5]

    def worker(t):
        def fn():
            torch.cuda.set_device(dev)
            s = torch.cuda.Stream(dev)
            for n in range(5):
                outs[t][n] = gdr.kkt_solve_host(xs[t]["k"], xs[t]["g"], xs[t]["beta"], output_dtype=torch.float32,
                                                stream=s.cuda_stream, device=dev)
            s.synchronize()
        return fn

    _run_threads([worker(0), worker(1)])
    for t in range(2):
        for o in outs[t]:
            assert torch.equal(o, refs[t])
    assert gdr.device_status() == gdr.GDR_OK
