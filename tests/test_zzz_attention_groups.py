"""Attention spans that straddle a 1024-position key group: the span's first
rows see no key of the last group, so that group's state is empty for them and
must contribute nothing to the merge across groups. 2040 + 16 also takes two
launches of 32 query rows (4 heads per kv head)."""
import pytest

from tests.test_gpu_full import attention_long_context

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.mark.parametrize("L,S", [(1020, 8), (2040, 16)])
def test_attention_span_straddles_a_key_group(L, S):
    attention_long_context(L, S)
