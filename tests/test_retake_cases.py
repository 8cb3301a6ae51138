"""CPU checks of the constructed retake rows (no GPU): each head's scores take
the path of the kernel's reference rule its parity test relies on."""
from retake_cases import reference_path, retake_scores


def test_head0_retakes_after_its_last_keys_passed():
    ev = reference_path(retake_scores(0).float().numpy())
    assert [e[:2] for e in ev] == [(2, "block")]
    assert 0.15 < ev[0][2] < 0.21          # the rescaled last keys keep ~18 %


def test_head1_fails_on_its_last_keys_alone():
    ev = reference_path(retake_scores(1).float().numpy())
    assert [e[:2] for e in ev] == [(2, "tail")]


def test_head2_moves_lazily_without_retake():
    assert reference_path(retake_scores(2).float().numpy()) == []


def test_whole_block_rule_retakes_heads_0_and_1():
    """The d = 128 kernel tests whole blocks only: both heads retake there."""
    for h in (0, 1):
        ev = reference_path(retake_scores(h).float().numpy(), tail_first=False)
        assert [e[:2] for e in ev] == [(2, "block")]
