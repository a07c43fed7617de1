"""The synthetic tensor lists have the stated shapes, flags and counts."""
import torch

import workloads as W


def test_full_size_counts():
    ae = W.action_expert()
    assert len(ae.tensors) == 144 and ae.trainable_numel == 302_008_320
    assert ae.effective_bytes_per_step() == 28 * 302_008_320
    hs = W.hsdp_shard_view()
    assert len(hs.tensors) == 256 and hs.trainable_numel == 6_476_136_448
    rep = [t for t in hs.tensors if not t.owned]
    assert len(rep) == 64 and all(t.name.endswith((".o", ".norm")) for t in rep)
    fl = W.flat()
    assert fl.trainable_numel == 1_500_000_256
    assert fl.effective_bytes_per_step() == 32 * 1_500_000_256
    lrs = [fl.group_lrs(t)[0] for t in range(1, 11)]
    assert lrs[0] == 1e-4 and all(a > b for a, b in zip(lrs, lrs[1:]))
    tn = W.tiny()
    assert tn.trainable_numel == 47_584 and sum(t.numel for t in tn.tensors) == 48_624


def test_many_small_distribution():
    ms = W.many_small()
    assert len(ms.tensors) == 20000
    sizes = [t.numel for t in ms.tensors]
    assert min(sizes) >= 1 and max(sizes) <= 65536
    frozen = sum(not t.trainable for t in ms.tensors)
    zero = sum(t.zero_grad for t in ms.tensors)
    assert frozen == 2000 and zero == 180
    assert all(t.trainable for t in ms.tensors if t.zero_grad)
    assert 90e6 < ms.trainable_numel < 125e6


def test_draws_are_seeded_and_per_tensor():
    w = W.SMALL["many_small"]()
    a = W.draw_grads(w, 1)
    b = W.draw_grads(w, 1)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    c = W.draw_grads(w, 2)
    assert not torch.equal(a[0], c[0])
    for t, g in zip(w.tensors, a):
        if t.zero_grad:
            assert not g.any()
    ae = W.SMALL["action_expert"]()
    g = W.draw_grads(ae, 1)
    assert all(x.dtype == torch.bfloat16 for x in g)
    p = W.draw_params(ae)
    assert all(x.dtype == torch.float32 for x in p)
