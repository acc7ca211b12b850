"""dd_lmhead_select_noalloc: the LM head + select for callers that cannot
allocate device memory (a host framework's pool or a fixed memory budget they
must not bypass, or latency-critical loops that cannot afford an allocation's
device synchronisation).  Its scratch is an array inside the library, so the
test checks that it agrees with the allocating entry point on two calls in a
row (the shared array keeps the previous call's contents) and that requests
beyond the array's size are refused.  Collected last on purpose."""
import numpy as np
import pytest

import synth
from tests.gpu_helpers import TOL_CONF, close, require_gpu, to_dev, torch

pytestmark = pytest.mark.gpu


def _inputs(rows, H, V, seed):
    x = to_dev(synth.make_activations(rows, H, seed=seed))
    w = to_dev(synth.make_activations(V, H, seed=seed + 1, std=synth.LOGIT_STD / np.sqrt(H)))
    return x, w


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


def test_noalloc_matches_allocating_entry_point_twice():
    require_gpu()
    from block_wise_masked_dd_b300.decoder import lmhead_select
    # two calls in a row, the second with a different shape, each checked
    # against dd_lmhead_select on the same inputs
    for rows, H, V, seed in [(256, 1024, 16384, 3), (96, 512, 8192, 4)]:
        x, w = _inputs(rows, H, V, seed)
        c_ref, a_ref = lmhead_select(x, w)
        torch.cuda.synchronize()
        conf, arg = _noalloc(x, w)
        close(conf.cpu().numpy(), c_ref.cpu().numpy(), TOL_CONF, "noalloc confidence")
        assert (arg.cpu().numpy() == a_ref.cpu().numpy()).all()


def test_noalloc_refuses_requests_beyond_its_scratch():
    require_gpu()
    from block_wise_masked_dd_b300 import binding as B
    x = torch.zeros((1, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.DDError) as e:
        # 4096 rows x 256 vocab tiles needs 12 MiB of partials
        B.dd_lmhead_select_noalloc(4096, 64, 65536, x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), 0)
    assert e.value.status == B.DD_ERR_INVALID_ARG
    assert "scratch" in B.dd_last_error()
