"""Speculative decoding with the model's MTP drafter (worklog Step 5 and
Step 6): the graph-size rule of the W4A4 card's serving notes (capture sizes
must be multiples of k + 1) and the step's shape check, on the CPU."""
import pytest

from nvfp4_quantized_moe_sigmoid_gb300.model import SpecDecodeStep, graph_sizes_not_multiple


def test_card_capture_sizes_fit_k3():
    # the W4A4 card's serving flags: cudagraph_capture_sizes for k = 3
    card = [4, 8, 16, 32, 40, 64, 96, 128, 192, 256, 384, 512, 768, 1024]
    assert graph_sizes_not_multiple(card, 3) == []


def test_sizes_that_are_not_multiples_of_k_plus_1_are_reported():
    assert graph_sizes_not_multiple([1, 2, 4, 8, 16, 24, 30, 32], 3) == [1, 2, 30]
    assert graph_sizes_not_multiple([3, 6, 8], 2) == [8]
    assert graph_sizes_not_multiple([5, 10], 4) == []


def test_verify_batch_must_be_k_plus_1():
    class Stack:  # the shape check runs before any device work
        T = 3

    with pytest.raises(ValueError):
        SpecDecodeStep(Stack(), None, 3)
