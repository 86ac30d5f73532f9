"""Host-side logic of the chunk-level scan: the automatic run count, the
workspace it needs and the argument checks (no GPU work)."""
import pytest

import kla_inputs


def _kla():
    import chunked_delta_rule_kla_gb300 as kla
    try:
        kla.load_library()
    except RuntimeError as e:
        pytest.skip(str(e))
    return kla


def test_auto_segments_policy():
    kla = _kla()
    L, Tr = kla_inputs.LONG, kla_inputs.TRAIN
    # long context, 16 heads: the carry alone would fill 32 of 152 SMs -> scan
    assert kla.kla_chunk_fwd_auto_segments(L.B, L.T, L.H, L.dk, L.dv) > 1
    # training shape, 64 heads x 2 column slices: enough parallelism already
    assert kla.kla_chunk_fwd_auto_segments(Tr.B, Tr.T, Tr.H, Tr.dk, Tr.dv) == 1
    # short sequences are never split below 32 chunks per run
    assert kla.kla_chunk_fwd_auto_segments(1, 64 * 63, 1, 128, 128) == 1
    assert kla.kla_chunk_fwd_auto_segments(1, 64 * 64, 1, 128, 128) == 2
    # fp32 I/O has no scan; invalid shapes give 0
    assert kla.kla_chunk_fwd_auto_segments(1, 1 << 17, 1, 128, 128, io=kla.KLA_IO_FP32) == 1
    assert kla.kla_chunk_fwd_auto_segments(1, 1024, 1, 96, 128) == 0


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128)])
def test_scan_workspace_formula(dk, dv):
    kla = _kla()
    B, T, H = 2, 1000, 3
    nchunks = -(-T // 64)
    base = kla.kla_chunk_fwd_scan_workspace_bytes(B, T, H, dk, dv, segments=1)
    rec = 8192 + 64 * dk * 2 + 768
    # d_k = d_v = 128 with few heads and no scan: one grid with two role counters
    # and per-chunk ready flags
    flags = -(-(2 + B * H * nchunks) * 4 // 256) * 256 if (dk, dv) == (128, 128) else 0
    assert base == 256 + B * H * nchunks * rec + flags
    assert base % 256 == 0
    base -= flags
    for segments in (2, 3, 5, 16, 40):
        seg_chunks = -(-nchunks // segments)
        nseg = -(-nchunks // seg_chunks)
        n = kla.kla_chunk_fwd_scan_workspace_bytes(B, T, H, dk, dv, segments=segments)
        assert n == base + B * H * nseg * dk * (2 * dv + dk) * 4
        assert n % 256 == 0
    assert kla.kla_chunk_fwd_workspace_bytes(B, T, H, dk, dv) == base + flags  # auto = 1 here


def test_scan_argument_errors():
    kla = _kla()
    lib = kla.load_library()
    args = [None] * 5 + [1e-6, None, None, None]
    # fp32 I/O supports no segmentation
    rc = lib.kla_chunk_fwd_scan(*args, 1, 128, 1, 128, 128, 64, kla.KLA_IO_FP32, 2, None, 0, None)
    assert rc == kla.KLA_ERR_UNSUPPORTED
    rc = lib.kla_chunk_fwd_scan(*args, 1, 128, 1, 128, 128, 64, kla.KLA_IO_BF16, -1, None, 0, None)
    assert rc == kla.KLA_ERR_INVALID_ARG
    assert kla.kla_chunk_fwd_scan_workspace_bytes(1, 128, 1, 128, 128, io=kla.KLA_IO_FP32, segments=2) == 0
    assert kla.kla_chunk_fwd_scan_workspace_bytes(1, 128, 1, 128, 128, segments=-1) == 0


@pytest.mark.parametrize("B,H,nchunks,extra", [
    (4, 19, 40, "flags"),      # 76 heads: prep lanes and carries in one grid
    (1, 77, 40, "handoff"),    # 77 heads, >= 32 chunks: chunk ranges hand the state over
    (1, 77, 31, "none"),       # 77 heads, < 32 chunks: one prep grid, then one carry grid
    (2, 68, 40, "handoff"),    # 136 heads: still chunk ranges
    (1, 137, 40, "none"),      # more heads: no ranges
])
def test_unsegmented_path_workspace(B, H, nchunks, extra):
    # d_k = d_v = 128 without a scan: the workspace names the path the call takes
    kla = _kla()
    T = 64 * nchunks - 5
    assert kla.kla_chunk_fwd_auto_segments(B, T, H, 128, 128) == 1
    n = kla.kla_chunk_fwd_workspace_bytes(B, T, H, 128, 128)
    base = 256 + B * H * nchunks * (8960 + 128 * 128)
    want = {"flags": -(-(2 + B * H * nchunks) * 4 // 256) * 256,
            "handoff": B * H * 128 * 128 * 4,
            "none": 0}[extra]
    assert n == base + want


def test_beta_mode_argument_errors():
    # an unknown step-size rule is refused before any device work
    kla = _kla()
    lib = kla.load_library()
    args = [None] * 5 + [1e-6, None, None, None]
    for bad in (-1, 2, 7):
        rc = lib.kla_chunk_fwd_ex(*args, 1, 128, 1, 128, 128, 64, kla.KLA_IO_BF16, bad, 0, None, 0,
                                  None)
        assert rc == kla.KLA_ERR_INVALID_ARG
        rc = lib.kla_decode_step_ex(None, None, None, None, None, 1e-6, None, None, 1, 1, 128, 128,
                                    kla.KLA_IO_BF16, bad, None)
        assert rc == kla.KLA_ERR_INVALID_ARG


def test_psd_feature_argument_errors():
    kla = _kla()
    lib = kla.load_library()
    # 16 (16+1)/2 = 136 features do not fit 128; 11 do not fit 64; d_out must be 64 or 128
    assert lib.kla_psd_features(None, None, 1, 16, 128, kla.KLA_IO_BF16, None) == kla.KLA_ERR_UNSUPPORTED
    assert lib.kla_psd_features(None, None, 1, 11, 64, kla.KLA_IO_BF16, None) == kla.KLA_ERR_UNSUPPORTED
    assert lib.kla_psd_features(None, None, 1, 4, 96, kla.KLA_IO_BF16, None) == kla.KLA_ERR_UNSUPPORTED
    assert lib.kla_psd_features(None, None, 1, 0, 64, kla.KLA_IO_BF16, None) == kla.KLA_ERR_INVALID_ARG
    assert lib.kla_psd_features(None, None, 1, 4, 64, kla.KLA_IO_BF16, None) == kla.KLA_ERR_INVALID_ARG
    assert lib.kla_psd_features(None, None, 0, 4, 64, kla.KLA_IO_BF16, None) == kla.KLA_OK
    assert lib.kla_psd_features_bwd(None, None, None, 1, 15, 64, kla.KLA_IO_FP32, None) == kla.KLA_ERR_UNSUPPORTED


def test_loglinear_levels_and_errors():
    kla = _kla()
    lib = kla.load_library()
    assert [kla.kla_loglinear_num_levels(T) for T in (1, 2, 64, 65, 4096, 131072)] == [1, 2, 7, 8, 13, 18]
    args = [None] * 6
    # too few levels for T = 100 (needs 8)
    rc = lib.kla_loglinear_fwd(*args, 7, 1e-6, None, 1, 100, 1, 128, 128, 64, kla.KLA_IO_BF16, 0,
                               None, 0, None)
    assert rc == kla.KLA_ERR_INVALID_ARG
    rc = lib.kla_loglinear_fwd(*args, 8, 1e-6, None, 1, 100, 1, 96, 128, 64, kla.KLA_IO_BF16, 0,
                               None, 0, None)
    assert rc == kla.KLA_ERR_UNSUPPORTED
    assert kla.kla_loglinear_workspace_bytes(1, 100, 1, 96, 128) == 0
    assert kla.kla_loglinear_workspace_bytes(1, 4096, 2, 128, 128) > 0


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128)])
def test_backward_workspace_formula(dk, dv):
    # per chunk-head: the prep record (gamma, beta, kk, T, Wk, U, P^T dO, L), the
    # start state and its gradient, W and dW; plus the error record
    kla = _kla()
    B, T, H = 2, 1000, 3
    items = B * H * -(-T // 64)
    rec = 3 * 64 + 64 * 64 + 64 * dk + 2 * 64 * dv + dk * dv
    body = 4 * items * (rec + 2 * dk * dv + 2 * 64 * dv)
    assert kla.kla_chunk_bwd_workspace_bytes(B, T, H, dk, dv) == 256 + -(-body // 256) * 256
    assert kla.kla_chunk_bwd_workspace_bytes(B, T, H, 96, dv) == 0
    assert kla.kla_chunk_bwd_workspace_bytes(1, 64, 65536, dk, dv) == 0     # B*H over 65535


@pytest.mark.parametrize("T", [1, 64, 65, 4096, 4097])
def test_loglinear_workspace_formula(T):
    # per chunk-head: gamma, Wk, U and the chunk's own output, then one state
    # slot per bit of the largest chunk index
    kla = _kla()
    B, H, dk, dv = 1, 2, 128, 64
    nch = -(-T // 64)
    bits = max(1, (nch - 1).bit_length())
    items = B * H * nch
    body = 4 * items * (64 + 64 * dk + 2 * 64 * dv + bits * dk * dv)
    assert kla.kla_loglinear_workspace_bytes(B, T, H, dk, dv) == 256 + -(-body // 256) * 256


def test_loglinear_decode_argument_errors():
    kla = _kla()
    lib = kla.load_library()
    args = [None] * 6
    # token 100 needs 1 + ceil(log2 101) = 8 levels; more than 32 are refused
    rc = lib.kla_loglinear_decode_step(*args, 7, 1e-6, None, 100, None, 1, 1, 128, 128, kla.KLA_IO_BF16, 0, None)
    assert rc == kla.KLA_ERR_INVALID_ARG
    rc = lib.kla_loglinear_decode_step(*args, 33, 1e-6, None, 100, None, 1, 1, 128, 128, kla.KLA_IO_BF16, 0, None)
    assert rc == kla.KLA_ERR_INVALID_ARG
    rc = lib.kla_loglinear_decode_step(*args, 8, 1e-6, None, 100, None, 1, 1, 96, 128, kla.KLA_IO_BF16, 0, None)
    assert rc == kla.KLA_ERR_UNSUPPORTED
    rc = lib.kla_loglinear_decode_step(*args, 8, 1e-6, None, -1, None, 1, 1, 128, 128, kla.KLA_IO_BF16, 0, None)
    assert rc == kla.KLA_ERR_INVALID_ARG
