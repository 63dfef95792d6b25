"""The top-k kernel sorts each lane's candidates with a fixed comparator
network before its warp-wide selection rounds (4 candidates per lane up to
128 experts, 8 above).  The networks are read from the kernel source and
checked exhaustively on 0/1 inputs (the 0-1 principle: a comparator network
that sorts every 0/1 sequence sorts every sequence).  No GPU needed."""

import itertools
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "nvfp4_token_quantized_gb300", "csrc", "kernels_route.cu")


def _networks():
    text = open(SRC, encoding="utf-8").read()
    body = text[text.index("void topk_warp_n("):]
    four = body[body.index("if constexpr (NE == 4)"):body.index("} else {")]
    net4 = [(int(a), int(b)) for a, b in re.findall(r"topk_cas\(key\[(\d+)\], key\[(\d+)\]\)", four)]
    m = re.search(r"constexpr int net\[(\d+)\]\[2\] = \{(.*?)\};", body, re.S)
    net8 = [(int(a), int(b)) for a, b in re.findall(r"\{(\d+), (\d+)\}", m.group(2))]
    assert len(net8) == int(m.group(1))
    return net4, net8


def _sorts_descending(net, n):
    for bits in itertools.product((0, 1), repeat=n):
        k = list(bits)
        for a, b in net:  # the larger key ends up at index a
            if k[a] < k[b]:
                k[a], k[b] = k[b], k[a]
        if k != sorted(bits, reverse=True):
            return False
    return True


def test_candidate_networks_sort_descending():
    net4, net8 = _networks()
    assert len(net4) == 5 and len(net8) == 19
    assert _sorts_descending(net4, 4)
    assert _sorts_descending(net8, 8)


def test_a_broken_network_is_caught():
    # the check itself must fail on a network with one comparator removed
    _, net8 = _networks()
    assert not _sorts_descending(net8[:-1], 8)
