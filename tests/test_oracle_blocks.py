"""The oracle's two-level indexer helpers (block-max keys and the candidate
block table) against numpy restatements of their definitions (no GPU)."""

import oracle
import oracle_pins as P


def test_amax8_matches_numpy_reshape_max():
    P.pin_amax8(oracle.load())


def test_sort_candidate_blocks_matches_numpy_sort():
    P.pin_sort_candidate_blocks(oracle.load())
