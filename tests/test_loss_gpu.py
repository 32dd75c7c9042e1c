"""spd_masked_token_loss on the GPU against the fp64 oracle: per-token losses,
the reproducible sum and count, the gradient rows, ignored tokens, a
vocabulary that is not a multiple of eight (scalar path) and a label outside
the vocabulary (reported in the device status word)."""
import numpy as np
import pytest
import torch

from oracle import loss as L

pytestmark = pytest.mark.gpu


def _ops():
    from sample_packing_document_gb300 import build, ops
    build.build()
    return ops


@pytest.mark.parametrize("T,V,seed", [(200, 50000, 0), (64, 1001, 1), (3, 7, 2), (1024, 4096, 3),
                                      (5, 1, 4), (9, 2, 5), (1, 8, 6), (1, 50000, 7),   # one class, two, one token
                                      (40, 131072, 8)])                               # larger than the smem row path
def test_loss_and_gradient_match_oracle(T, V, seed):
    ops = _ops()
    g = torch.Generator().manual_seed(seed)
    logits = (torch.randn((T, V), generator=g) * 3).to(torch.bfloat16)
    rng = np.random.default_rng(seed)
    labels = rng.integers(0, V, size=T).astype(np.int32)
    labels[rng.random(T) < 0.25] = -100
    x = logits.float().numpy()
    want_tok = L.token_losses(x, labels)
    s, n, _ = L.masked_loss(x, labels)
    scale = 1.0 / max(n, 1)
    dl = torch.empty((T, V), dtype=torch.bfloat16, device="cuda")
    tok, ssum, cnt = ops.masked_token_loss(logits.cuda(), torch.tensor(labels, device="cuda"), dlogits=dl,
                                           grad_scale=scale)
    torch.cuda.synchronize()
    assert int(cnt.item()) == n
    assert np.allclose(tok.cpu().numpy(), want_tok, rtol=1e-5, atol=1e-4)
    assert float(ssum.item()) == pytest.approx(s, rel=1e-5, abs=1e-3)
    want_g = L.logits_grad(x, labels, scale)
    got_g = dl.float().cpu().numpy()
    # bf16 rounding of each gradient entry (half an ulp) plus the fp32 softmax
    assert np.all(np.abs(got_g - want_g) <= 2.0 ** -8 * np.abs(want_g) + 1e-6 * scale)


def test_all_ignored_and_bad_label():
    ops = _ops()
    logits = torch.zeros((4, 16), dtype=torch.bfloat16, device="cuda")
    tok, ssum, cnt = ops.masked_token_loss(logits, torch.full((4,), -100, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert float(ssum.item()) == 0.0 and int(cnt.item()) == 0 and not tok.any()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    labels = torch.tensor([3, 16, -100, 5], dtype=torch.int32, device="cuda")   # 16 is outside [0, 16)
    tok, ssum, cnt = ops.masked_token_loss(logits, labels, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -1 and int(cnt.item()) == 2
    assert float(ssum.item()) == pytest.approx(2 * np.log(16.0), rel=1e-6)   # uniform logits: log V each
