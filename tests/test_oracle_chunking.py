"""Pins for the pipeline chunk-size rule (no GPU): the chunk sizes the page prints.

strata #1441, "Prompt chunks sized for a layer split's pipeline": the table of
prompt tok/s lists the chunk the rule chose on four stages with b/a = 1024 for
four prompt lengths, and the summary gives the same sizes in words.
"""

import pytest

from oracle.chunking import pipeline_chunk


@pytest.mark.parametrize("n,chunk", [(2013, 1024), (3865, 1024), (10041, 2048), (28998, 3328)])
def test_printed_chunks_on_four_stages(n, chunk):
    assert pipeline_chunk(n, cap=8192, stages=4) == chunk


def test_rule_properties():
    # one stage keeps the whole prompt (up to the cap); the result stays on the grid within [512, cap]
    assert pipeline_chunk(10041, cap=8192, stages=1) == 8192
    assert pipeline_chunk(300, cap=8192, stages=4) == 300
    for n in range(600, 40000, 997):
        c = pipeline_chunk(n, cap=4096, stages=4)
        assert c == n or (c % 256 == 0 and 512 <= c <= 4096)
    # the chunk grows with the square root of the prompt: 4x the tokens, about 2x the chunk
    assert pipeline_chunk(4 * 10041, cap=1 << 20, stages=4) in range(3840, 4352, 256)
