"""The one-copy staging of a step's host inputs (host logic, no GPU)."""

import torch

from paged_gqa_decode_rope_gb300 import ops


def test_views_are_aligned_disjoint_and_round_trip():
    specs = {"q": ((3, 64, 128), torch.bfloat16), "positions": ((3,), torch.int32),
             "slot_mapping": ((3,), torch.int64), "block_table": ((3, 5), torch.int32),
             "odd": ((7,), torch.uint8)}
    st = ops.HostInputs(specs, device="cpu")
    spans = []
    for name, (shape, dtype) in specs.items():
        off, nbytes, _, _ = st.offsets[name]
        assert off % 256 == 0
        assert tuple(st.host[name].shape) == shape and st.host[name].dtype == dtype
        spans.append((off, off + nbytes))
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))
    assert st.nbytes >= spans[-1][1] and st.nbytes % 256 == 0
    g = torch.Generator().manual_seed(0)
    vals = {n: (torch.randn(shape, generator=g).to(dtype) if dtype.is_floating_point
                else torch.randint(0, 100, shape, generator=g).to(dtype))
            for n, (shape, dtype) in specs.items()}
    for n, v in vals.items():
        st.host[n].copy_(v)
    dev = st.upload()
    for n, v in vals.items():
        assert torch.equal(dev[n], v)
