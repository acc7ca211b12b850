"""dd_lmhead_select_noalloc: the LM head + select for callers that cannot
allocate device memory (a host framework's pool or a fixed memory budget they
must not bypass, or latency-critical loops that cannot afford an allocation's
device synchronisation).  Its scratch is an array inside the library, so the
tests check it against the oracle and against the allocating entry point on
calls in a row (the shared array keeps the previous call's contents), at the
largest request the array holds, that a request one row over is refused, and
that a call after the warm-up leaves the device's free memory unchanged.
Collected last on purpose."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import TOL_CONF, close, require_gpu, to_dev, torch

pytestmark = pytest.mark.gpu

# rows * (vocab / 256) at most 698944: three fp32 arrays of that many entries
# (each rounded up to 256 bytes) after a 256-byte status word fill 8 MiB
LIMIT_ROW_TILES = 698944


def _inputs(rows, H, V, seed):
    xb = synth.make_activations(rows, H, seed=seed)
    wb = synth.make_activations(V, H, seed=seed + 1, std=synth.LOGIT_STD / np.sqrt(H))
    return xb, wb, to_dev(xb), to_dev(wb)


def _noalloc(x, w):
    from block_wise_masked_dd_b300 import binding as B
    rows, H = x.shape
    V = w.shape[0]
    conf = torch.empty(rows, dtype=torch.float32, device="cuda")
    arg = torch.empty(rows, dtype=torch.int32, device="cuda")
    B.dd_lmhead_select_noalloc(rows, H, V, x.data_ptr(), w.data_ptr(), conf.data_ptr(), arg.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return conf, arg


def test_noalloc_matches_oracle_and_allocating_entry_point_twice():
    require_gpu()
    from block_wise_masked_dd_b300.decoder import lmhead_select
    # two calls in a row, the second with a different shape, each checked
    # against the oracle's LM head + select and against dd_lmhead_select
    for rows, H, V, seed in [(256, 1024, 16384, 3), (96, 512, 8192, 4)]:
        xb, wb, x, w = _inputs(rows, H, V, seed)
        conf, arg = _noalloc(x, w)
        c, a = conf.cpu().numpy(), arg.cpu().numpy()
        want_c, want_a, logits = oracle.lm_head_select(synth.bf16_bits_to_f32(xb), synth.bf16_bits_to_f32(wb))
        close(c, want_c, TOL_CONF, "noalloc confidence vs oracle")
        tie = oracle.top2_gap(logits) < oracle.TIE_LOGIT_GAP
        assert ((a == want_a) | tie).all(), f"argmax differs from the oracle at rows {np.nonzero((a != want_a) & ~tie)[0][:8]}"
        c_ref, a_ref = lmhead_select(x, w)
        torch.cuda.synchronize()
        close(c, c_ref.cpu().numpy(), TOL_CONF, "noalloc confidence vs dd_lmhead_select")
        assert (a == a_ref.cpu().numpy()).all()


def test_noalloc_largest_request_and_one_row_over():
    require_gpu()
    from block_wise_masked_dd_b300 import binding as B
    from block_wise_masked_dd_b300.decoder import lmhead_select
    V, H = 65536, 64
    rows = LIMIT_ROW_TILES // (V // 256)          # 2730 rows: the partials nearly fill the array
    _, _, x, w = _inputs(rows, H, V, 5)
    conf, arg = _noalloc(x, w)
    c_ref, a_ref = lmhead_select(x, w)
    torch.cuda.synchronize()
    close(conf.cpu().numpy(), c_ref.cpu().numpy(), TOL_CONF, "noalloc confidence at the size limit")
    assert (arg.cpu().numpy() == a_ref.cpu().numpy()).all()
    with pytest.raises(B.DDError) as e:
        B.dd_lmhead_select_noalloc(rows + 1, H, V, x.data_ptr(), w.data_ptr(), conf.data_ptr(), arg.data_ptr(), 0)
    assert e.value.status == B.DD_ERR_INVALID_ARG
    assert "scratch" in B.dd_last_error()


def test_noalloc_refuses_requests_beyond_its_scratch():
    require_gpu()
    from block_wise_masked_dd_b300 import binding as B
    x = torch.zeros((1, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.DDError) as e:
        # 4096 rows x 256 vocab tiles needs 12 MiB of partials
        B.dd_lmhead_select_noalloc(4096, 64, 65536, x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), 0)
    assert e.value.status == B.DD_ERR_INVALID_ARG
    assert "scratch" in B.dd_last_error()


def test_noalloc_call_after_warm_up_allocates_nothing():
    require_gpu()
    _, _, x, w = _inputs(128, 512, 8192, 6)
    conf = torch.empty(128, dtype=torch.float32, device="cuda")
    arg = torch.empty(128, dtype=torch.int32, device="cuda")
    from block_wise_masked_dd_b300 import binding as B
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        B.dd_lmhead_select_noalloc(128, 512, 8192, x.data_ptr(), w.data_ptr(), conf.data_ptr(), arg.data_ptr(), stream)
        torch.cuda.synchronize()
    call()                                   # warm-up: may load the module and create the array
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        call()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory moved by {free0 - free1} bytes across calls after the warm-up"
