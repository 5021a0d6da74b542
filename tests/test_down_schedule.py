"""Host-side restatement of the down-projection tile schedule (row-block major for at most 12
expert slots, expert major above), checked for the invariants the kernel relies on: every tile
is taken exactly once, the producer's weight addresses and the consumer's (expert, k block)
walk agree, each output row block's counter gains exactly nv * kb_i tiles, and a CTA's range
spans few experts (the SwiGLU rows it stages). Pure integer arithmetic, no GPU."""
import pytest

RB_MAJOR_MAX = 12  # kDRowMajorMax


def _range_lo(T, c, G):
    return T * c // G


def _walk(n_rb_d, kb_i, nv, G):
    rbm = nv <= RB_MAJOR_MAX
    tpe = kb_i if rbm else n_rb_d * kb_i
    kbs = nv * kb_i if rbm else kb_i
    T = n_rb_d * nv * kb_i
    seen, cnt, span = set(), [0] * n_rb_d, 0
    for c in range(G):
        t0, t1 = _range_lo(T, c, G), _range_lo(T, c + 1, G)
        if t1 <= t0:
            continue
        # producer cursor: (expert slot, tile index within that expert's [rb][kb] weights)
        if rbm:
            rb = t0 // kbs
            k = t0 - rb * kbs
            u, r = k // tpe, k % tpe
            addr = [u, rb * kb_i + r]
        else:
            addr = [t0 // tpe, t0 % tpe]
        # consumer walk
        seg, kb = t0 // kbs, t0 % kbs
        v = kb // tpe if rbm else t0 // tpe
        rv = kb - v * tpe if rbm else t0 - v * tpe
        kx, xj = rv % kb_i, 0
        s0 = t0 // tpe
        nst = min((t1 - 1) // tpe - s0 + 1, nv)
        staged = [(s0 % nv + j) % nv for j in range(nst)]
        span = max(span, nst)
        for _ in range(t0, t1):
            pu, pr = addr
            assert pu == v and staged[xj] == v and pr % kb_i == kx
            key = (pu, pr // kb_i, pr % kb_i)
            assert key not in seen
            seen.add(key)
            assert (seg if rbm else seg % n_rb_d) == pr // kb_i  # counter = the tile's row block
            cnt[pr // kb_i] += 1
            # producer advance
            if rbm:
                if (pr % kb_i) + 1 == tpe:
                    nu, nrb = pu + 1, pr // kb_i
                    if nu == nv:
                        nu, nrb = 0, nrb + 1
                    addr = [nu, nrb * kb_i]
                else:
                    addr = [pu, pr + 1]
            else:
                addr = [pu + 1, 0] if pr + 1 == tpe else [pu, pr + 1]
            # consumer advance
            kb += 1
            if kb == kbs:
                kb, seg = 0, seg + 1
            kx = 0 if kx + 1 == kb_i else kx + 1
            rv += 1
            if rv == tpe:
                rv = 0
                v = 0 if v + 1 == nv else v + 1
                xj = 0 if xj + 1 == nv else xj + 1
    assert len(seen) == T
    assert cnt == [nv * kb_i] * n_rb_d
    return rbm, span


@pytest.mark.parametrize("n_rb_d,kb_i", [(32, 12), (4, 2), (2, 1)])
@pytest.mark.parametrize("nv", [1, 2, 5, 9, 12, 13, 17, 33, 65])
def test_down_schedule_invariants(n_rb_d, kb_i, nv):
    rbm, span = _walk(n_rb_d, kb_i, nv, 152)
    assert rbm == (nv <= RB_MAJOR_MAX)
    if n_rb_d == 32:  # the 8-layer stack: a CTA stages at most 4 experts' SwiGLU rows
        assert span <= 4
