"""The hybrid layer pattern used for the model-ordered verify step, checked
against the counts the technical-report summary states (section
"MiMo-V2-Flash Model Architecture" and its hyper-parameter paragraph):
48 layers, 39 SWA and 9 GA, M = 8 blocks of 5 SWA layers then one GA layer,
and the first layer of the stack uses global attention."""
import synth


def test_hybrid_layer_pattern_matches_the_stated_counts():
    kinds = synth.hybrid_layer_kinds()
    assert len(kinds) == 48
    assert kinds.count("swa") == 39 and kinds.count("ga") == 9
    assert kinds[0] == "ga"
    for blk in range(8):   # every block of six ends with its GA layer
        assert kinds[6 * blk + 5] == "ga"
    # outside the first layer, every block is five SWA layers then one GA layer
    assert kinds[1:6] == ["swa"] * 4 + ["ga"]
    for blk in range(1, 8):
        assert kinds[6 * blk:6 * blk + 6] == ["swa"] * 5 + ["ga"]
