"""Host-side checks of the seeded input generators (no GPU): shapes, dtypes, determinism and the structure the
workloads promise (the WY chunk matrices are unit lower-triangular per chunk, chunks starting at each
sequence's first row)."""
import numpy as np
import torch

from chunkwise_gated_linear_chunked_gb300.inputs import WORKLOADS, make_inputs, make_wy_inputs, stored_numpy


def test_forward_inputs_are_seeded_and_shaped():
    a = make_inputs("bf16", B=2, T=70, H=3, K=64, V=128, h0=True, seed=5)
    b = make_inputs("bf16", B=2, T=70, H=3, K=64, V=128, h0=True, seed=5)
    assert a.q.shape == (2, 70, 3, 64) and a.v.shape == (2, 70, 3, 128) and a.h0.shape == (2, 3, 64, 128)
    assert a.q.dtype == torch.bfloat16 and a.h0.dtype == torch.float32
    assert all(torch.equal(x, y) for x, y in zip((a.q, a.k, a.v, a.g, a.h0), (b.q, b.k, b.v, b.g, b.h0)))
    assert float(a.g.float().max()) <= 0.0          # log-decays
    v = make_inputs("f32", H=2, K=64, V=64, lengths=[3, 0, 65], seed=1)
    assert v.B == 1 and v.T == 68 and v.N == 3 and v.cu_seqlens.tolist() == [0, 3, 3, 68]


def test_wy_inputs_structure():
    lengths = [5, 64, 0, 70, 1]
    x = make_wy_inputs("bf16", H=2, HV=4, K=64, V=128, BT=16, lengths=lengths, seed=3)
    rows = sum(lengths)
    assert x.k.shape == (1, rows, 2, 64) and x.v.shape == (1, rows, 4, 128) and x.A.shape == (1, rows, 4, 16)
    assert x.beta.shape == (1, rows, 4) and x.g.shape == (1, rows, 4) and x.g.dtype == torch.float32
    assert float(x.g.max()) <= 0.0 and float(x.g.min()) >= -4.0
    assert 0.0 < float(x.beta.float().min()) and float(x.beta.float().max()) < 1.0
    A = x.A.float()[0].numpy()
    starts = np.concatenate([[0], np.cumsum(lengths)])
    for s0, s1 in zip(starts[:-1], starts[1:]):
        for t in range(s0, s1):
            p = (t - s0) % 16
            assert np.all(A[t, :, p] == 1.0)                 # unit diagonal at the row's chunk position
            assert np.all(A[t, :, p + 1:] == 0.0)            # nothing above it
    d = make_wy_inputs("f32", B=2, T=40, H=1, HV=1, K=64, V=64, BT=32, seed=4)
    pos = np.tile(np.arange(40) % 32, 2)
    Ad = d.A[..., 0, :].reshape(80, 32).numpy()
    assert np.all(Ad[np.arange(80), pos] == 1.0)


def test_stored_numpy_keeps_the_stored_words():
    x = torch.tensor([1.0, -2.5, 3.140625], dtype=torch.bfloat16)
    w = stored_numpy(x)
    assert w.dtype == np.uint16 and w.tolist() == [0x3F80, 0xC020, 0x4049]
    assert stored_numpy(x.float()).dtype == np.float32 and stored_numpy(x.half()).dtype == np.float16


def test_workload_table_names_what_it_holds():
    for name, w in WORKLOADS.items():
        assert w.name == name and w.note
