"""Handles used from several host threads at once give what they give one at a time.

Each thread owns a handle of a different shape (other router exchange modes, FFN tilings
and staging plans, so the library's per-device launch caches and per-kernel shared-memory
limits are set concurrently) and runs forward passes on its own stream; every output must
equal the same handle's single-threaded result bit for bit.
"""
import threading

import pytest
import torch

from gen import LayerShape, make_inputs
import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


SHAPES = [
    (LayerShape("thr-a", 2, 300, 256, 384, 8, 1.0), 1),
    (LayerShape("thr-b", 1, 900, 128, 128, 200, 1.0), 1),
    (LayerShape("thr-c", 1, 600, 128, 128, 1100, 1.0), 1),
    (LayerShape("thr-d", 1, 700, 512, 1024, 4, 1.0), 1),
    (LayerShape("thr-e", 1, 500, 128, 256, 40, 1.0), 2),  # top-2: the logits pass's staging
]


def _run(layer, inp, stream, reps):
    outs = []
    with torch.cuda.stream(stream):
        for _ in range(reps):
            y, r = layer.forward(inp["x"], inp["Wr"], inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"],
                                 stream=stream)
            outs.append((y.clone(), r.expert.clone(), r.gate.clone()))
    stream.synchronize()
    return outs


def test_concurrent_handles_match_sequential():
    cases = []
    for shape, k in SHAPES:
        inp = make_inputs(shape, 17, "cuda", router_bias_std=0.1)
        layer = P.make_layer(shape, top_k=k)
        cases.append((layer, inp, torch.cuda.Stream()))
    ref = [_run(layer, inp, st, 1)[0] for layer, inp, st in cases]

    results = [None] * len(cases)
    errors = []

    def work(i):
        try:
            layer, inp, st = cases[i]
            results[i] = _run(layer, inp, st, 3)
        except Exception as exc:  # reported below, in the main thread
            errors.append(exc)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, (shape, _) in enumerate(SHAPES):
        for y, e, g in results[i]:
            assert torch.equal(y, ref[i][0]) and torch.equal(e, ref[i][1]) and torch.equal(g, ref[i][2]), shape.name
    for layer, _, _ in cases:
        layer.sync_status()
