"""Token-budget accounting of the SparseEngine settings tables.

TEST INFRASTRUCTURE (see the package docstring).

[SparseEngine: Sparse-First Inference Engine, Table 10 caption]: selected
budgets exclude separately listed sink and recent tokens, so the tokens a
method keeps are selected + sink + recent (the "total" column of Tables 9-11).
Quest selects whole 16-token pages (Tables 8, 9, 11), so a selected budget of
T tokens is T / 16 pages (Table 10: 2,048 selected = 128 pages).
"""


def total_kept_tokens(selected: int, sink: int, recent: int) -> int:
    return selected + sink + recent


def selected_pages(selected_tokens: int, page_size: int = 16) -> int:
    if selected_tokens % page_size:
        raise ValueError("a page-granular budget must be a whole number of pages")
    return selected_tokens // page_size
