"""How matmul hands its operands to bil_linear_gemm (host logic, no GPU): an operand
whose K dimension has unit stride goes as K-major, one whose row dimension has unit
stride (a transposed view of a row-major matrix) as MN-major, each with the row stride
of its stored rows; anything else, or rows that are not 16-byte multiples, goes as a
padded K-major copy with the same elements."""
import torch

from invariant_token_log_gb300 import _lib
from invariant_token_log_gb300.linear import _rows_over_k

K, MN = _lib.LAYOUT_K_MAJOR, _lib.LAYOUT_MN_MAJOR


def _aligned(rows, cols, dtype=torch.bfloat16):
    return torch.randn(rows, cols).to(dtype)


def _elements(x, layout, ld, rows, k):
    """The [rows, k] matrix bil_linear_gemm reads from x's storage with this layout."""
    flat = x.as_strided((x.untyped_storage().nbytes() // x.element_size(),), (1,), 0)
    base = x.storage_offset()
    i = torch.arange(rows).view(-1, 1)
    kk = torch.arange(k).view(1, -1)
    idx = base + (i * ld + kk if layout == K else kk * ld + i)
    return flat[idx]


def test_a_row_major_operand_is_k_major():
    a = _aligned(40, 64)
    x, layout, ld = _rows_over_k(a, 1)
    assert (layout, ld) == (K, 64) and x.data_ptr() == a.data_ptr()
    assert torch.equal(_elements(x, layout, ld, 40, 64), a)


def test_a_transposed_view_is_mn_major():
    s = _aligned(64, 40)          # stored [k, m]
    a = s.t()                     # [m, k] view
    x, layout, ld = _rows_over_k(a, 1)
    assert (layout, ld) == (MN, 40) and x.data_ptr() == s.data_ptr()
    assert torch.equal(_elements(x, layout, ld, 40, 64), a)


def test_b_as_matmul_takes_it():
    # matmul's b is [k, n]; B's rows are its columns
    b = _aligned(64, 24)          # row-major [k, n]: MN-major B
    x, layout, ld = _rows_over_k(b, 0)
    assert (layout, ld) == (MN, 24)
    assert torch.equal(_elements(x, layout, ld, 24, 64), b.t())
    bt = _aligned(24, 64).t()     # transposed view of row-major [n, k]: K-major B
    x, layout, ld = _rows_over_k(bt, 0)
    assert (layout, ld) == (K, 64)
    assert torch.equal(_elements(x, layout, ld, 24, 64), bt.t())


def test_rows_of_odd_length_and_strided_views_are_copied():
    a = _aligned(10, 36)          # 72-byte rows: not a 16-byte multiple
    x, layout, ld = _rows_over_k(a, 1)
    assert layout == K and ld % 8 == 0 and x.data_ptr() != a.data_ptr()
    assert torch.equal(x, a)
    big = _aligned(20, 64)
    v = big[::2, ::2]             # no unit-stride dimension
    x, layout, ld = _rows_over_k(v, 1)
    assert layout == K and torch.equal(x, v)


def test_single_rows_and_columns():
    a = _aligned(1, 64)           # one row: K-major, its row stride at least k
    x, layout, ld = _rows_over_k(a, 1)
    assert layout == K and ld >= 64
    assert torch.equal(_elements(x, layout, ld, 1, 64), a)
    s = _aligned(64, 8)[:, :1]    # [k, 1] column of a row-major [k, 8]: MN-major A of one row
    x, layout, ld = _rows_over_k(s.t(), 1)
    assert (layout, ld) == (MN, 8)
    assert torch.equal(_elements(x, layout, ld, 1, 64), s.t())
