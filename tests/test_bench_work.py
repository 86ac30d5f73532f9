"""The bench's algorithmic work models (the numerators of every roofline
fraction it reports), recomputed from the tensors each call must touch."""
import bench
import kla_inputs


def test_prefill_bytes_of_the_training_shape():
    c = kla_inputs.TRAIN
    w = bench.prefill_work(c)
    toks = c.B * c.T * c.H
    # q, k, v, o in bf16 and g, eta in fp32 once per token-head; hT once per head
    want = toks * (2 * (2 * c.dk + 2 * c.dv) + 2 * 4) + c.B * c.H * c.dk * c.dv * 4
    assert w["bytes"] == want
    assert round(w["bytes"] / 1e6, 1) == 274.7


def test_backward_bytes_and_flops():
    c = kla_inputs.TRAIN
    w = bench.backward_work(c)
    toks = c.B * c.T * c.H
    # read q, k, v, dO (bf16), g, eta; write dq, dk, dv (bf16), dg, deta; dhT in, dh0 out
    per_tok = 2 * (c.dk + c.dk + c.dv + c.dv) + 2 * (c.dk + c.dk + c.dv) + 4 * 4
    assert w["bytes"] == toks * per_tok + 2 * c.B * c.H * c.dk * c.dv * 4
    # products per chunk of 64, divided by its 64 tokens:
    C = 64
    prep = 2 * (C * C * c.dk + C * c.dk * C + C * c.dv * C + C * C * c.dk + C * c.dv * C)
    carries = 2 * (2 * C * c.dk * c.dv + 3 * C * c.dk * c.dv)
    grads = 2 * (6 * C * C * c.dk + 4 * C * C * c.dv + 4 * C * c.dk * c.dv)
    assert w["flops"] == toks * (prep + carries + grads) // C
    assert round(w["bytes"] / 1e6, 1) == 482.3 and round(w["flops"] / 1e9, 1) == 141.7


def test_loglinear_and_deltakata_bytes():
    c = kla_inputs.TRAIN
    toks = c.B * c.T * c.H
    L = 13
    w = bench.loglinear_work(c, L)
    assert w["bytes"] == toks * (2 * (2 * c.dk + 2 * c.dv) + 8 + 4 * L)
    p = 15
    wd = bench.deltakata_work(c, p)
    assert wd["bytes"] == toks * (2 * (2 * p + 2 * c.dv) + 8) + c.B * c.H * c.dk * c.dv * 4


def test_decode_bytes():
    c = kla_inputs.DECODE
    w = bench.decode_work(c)
    heads = c.B * c.H
    # the fp32 state read and written, q, k, v, o in bf16, g and eta
    assert w["bytes"] == heads * (2 * c.dk * c.dv * 4 + 2 * (2 * c.dk + 2 * c.dv) + 8)
    assert round(w["bytes"] / 1e6, 1) == 135.3


def test_loglinear_decode_bytes_against_a_simulated_bucket_set():
    # replay the buckets token by token (the set of non-empty levels as the
    # decode step defines it) and count the state tiles read and written
    import bench
    B, H, dk, dv, L, steps, esz = 2, 3, 128, 64, 11, 300, 2
    tile = dk * dv * 4
    nonempty = set()
    want = 0
    for t in range(steps):
        reads = writes = 0
        if t > 0:
            reads = len(nonempty)                    # every non-empty level takes the transition
            b = (t & -t).bit_length() - 1
            assert b + 1 not in nonempty
            merged = {l for l in nonempty if l <= b}
            writes = len(nonempty - merged) + 1       # the rest written back, the merge target written
            nonempty = (nonempty - merged) | {b + 1}
        writes += 1                                   # the new level 0
        nonempty.add(0)
        want += B * H * ((reads + writes) * tile + esz * (2 * dk + 2 * dv) + 8 + 4 * L)
    assert bench.loglinear_decode_bytes(B, H, dk, dv, L, steps, esz) == want
