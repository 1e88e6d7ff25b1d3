"""Host-side helpers of the binding (no GPU): the per-CTA occupancy summary
behind the bench's schedule comparison, and the staged-page count of the
E4M3 prefill."""

import numpy as np
import torch

from paged_gqa_decode_rope_gb300 import ops


def test_cta_occupancy_on_hand_made_records():
    # [start ns, end ns, SM id] per CTA; CTA rows with end 0 did not run
    rec = torch.tensor([[0, 100, 0],      # SM 0 busy 0..100 and 100..160
                        [100, 160, 0],
                        [10, 200, 1],     # SM 1 busy 10..200 (the last end overall)
                        [20, 120, 2],     # SM 2 busy 20..120
                        [0, 0, 3]],       # never ran
                       dtype=torch.int64)
    occ = ops.cta_occupancy(rec)
    span = 200 - 0
    busy = (100 + 60) + 190 + 100
    assert occ["sms"] == 3 and occ["ctas"] == 4
    assert abs(occ["span_us"] - span / 1e3) < 1e-9
    assert abs(occ["occupancy"] - round(busy / (3 * span), 4)) < 1e-12
    # tail idle: mean over SMs of (last end overall - that SM's last end)
    assert abs(occ["tail_idle_us"] - round(((200 - 160) + 0 + (200 - 120)) / 3 / 1e3, 2)) < 1e-12


def test_pages_for_counts_ceil_of_lengths():
    assert ops.PrefillAttention.pages_for([]) == 0
    assert ops.PrefillAttention.pages_for([0, 1, 63, 64, 65, 128, 129]) == 0 + 1 + 1 + 1 + 2 + 2 + 3
    lens = np.random.default_rng(0).integers(0, 10000, 500)
    assert ops.PrefillAttention.pages_for(lens) == int(sum((int(L) + 63) // 64 for L in lens))
