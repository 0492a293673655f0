"""The seeded paged-cache layout (inputs.paged_cache) on CPU: every cached
token lands in slot t mod p of its request's (t // p)-th page, the pages
are a seeded permutation of the pool, table entries past a request's last
page are -1, and every slot no token uses holds the fill value."""

import torch

from linear_attention_diffusion_feature_b300 import inputs


def _layout(lens, pt, spare=3, seed=5):
    H, d = 2, 8
    kc = inputs.draw(1, (sum(lens), H, d), torch.float32)
    vc = inputs.draw(2, (sum(lens), H, d), torch.float32)
    return kc, vc, inputs.paged_cache(seed, kc, vc, lens, pt, spare_pages=spare)


def test_tokens_land_in_their_slots():
    lens = [0, 5, 64, 70, 33]
    pt = 32
    kc, vc, (kp, vp, table, plen) = _layout(lens, pt)
    assert plen.tolist() == lens
    row = 0
    for b, P in enumerate(lens):
        for t in range(P):
            page = int(table[b, t // pt])
            assert torch.equal(kp[page, t % pt], kc[row + t])
            assert torch.equal(vp[page, t % pt], vc[row + t])
        row += P


def test_table_pages_are_distinct_and_padded():
    lens = [0, 5, 64, 70, 33]
    pt = 16
    _, _, (kp, _, table, _) = _layout(lens, pt, spare=4)
    n_pages = [-(-P // pt) for P in lens]
    assert kp.shape[0] == sum(n_pages) + 4
    assert table.shape == (len(lens), max(n_pages))
    used = []
    for b, n in enumerate(n_pages):
        used += table[b, :n].tolist()
        assert (table[b, n:] == -1).all()
    assert len(set(used)) == len(used) and all(0 <= p < kp.shape[0] for p in used)


def test_unused_slots_hold_the_fill():
    lens = [5, 40]
    pt = 32
    kc, _, (kp, _, table, _) = _layout(lens, pt, spare=2)
    written = torch.zeros(kp.shape[:2], dtype=torch.bool)
    for b, P in enumerate(lens):
        for t in range(P):
            written[int(table[b, t // pt]), t % pt] = True
    assert torch.isnan(kp[~written]).all()
    assert not torch.isnan(kp[written]).any()
    assert int(written.sum()) == sum(lens)


def test_layout_is_seeded():
    a = _layout([10, 50], 32, seed=7)[2][2]
    b = _layout([10, 50], 32, seed=7)[2][2]
    c = _layout([10, 50], 32, seed=8)[2][2]
    assert torch.equal(a, b)
    assert not torch.equal(a, c)
